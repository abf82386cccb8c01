"""Plant plausible mistakes in copies of the oracle and check that at least one
pin rejects each (CPU only; the real oracle is untouched)."""
import os

import pytest

import oracle
from oracle import build as obuild
import oracle_pins

SRC = open(obuild.SRC).read()

# (name, original text, planted text)
MUTANTS = [
    ("exponent_bias", "(int)expo - 25", "(int)expo - 24"),
    ("subnormal_scale", "pow2i(-24)", "pow2i(-25)"),
    ("sign_dropped", "return sign ? -v : v;", "return v;"),
    ("last_term_dropped", "for (int64_t k = 0; k < K; ++k)", "for (int64_t k = 0; k + 1 < K; ++k)"),
    ("b_row_stride", "const uint16_t *b_row = B + b * sB + j * ldb;",
     "const uint16_t *b_row = B + b * sB + j;"),
    ("a_batch_stride", "const uint16_t *a_row = A + b * sA + i * lda;",
     "const uint16_t *a_row = A + b * sB + i * lda;"),
    ("abs_missing", "aacc += fabs(p);", "aacc += p;"),
    ("float_accumulator", "double acc = 0.0, aacc = 0.0;", "float acc = 0.0f; double aacc = 0.0;"),
    ("sampled_ij_swapped", "iidx[s] * lda", "jidx[s] * lda"),
    ("product_sign", "oracle_half_to_double(a_row[k]) * oracle_half_to_double(b_row[k])",
     "-oracle_half_to_double(a_row[k]) * oracle_half_to_double(b_row[k])"),
    ("bf16_exponent_bias", "(int)expo - 134", "(int)expo - 133"),
    ("bf16_subnormal_scale", "pow2i(-133)", "pow2i(-134)"),
    ("bf16_fraction_width", "const unsigned frac = h & 0x7fu;", "const unsigned frac = h & 0x3fu;"),
    ("bf16_last_term_dropped", "oracle_bf16_to_double(a_row[k]) * oracle_bf16_to_double(b_row[k])",
     "(k + 1 < K ? oracle_bf16_to_double(a_row[k]) * oracle_bf16_to_double(b_row[k]) : 0.0)"),
    ("e4m3_exponent_bias", "(int)expo - 10", "(int)expo - 9"),
    ("e4m3_subnormal_scale", "v = (double)frac * pow2i(-9);", "v = (double)frac * pow2i(-10);"),
    ("e4m3_nan_as_value", "if (expo == 15 && frac == 7) {", "if (expo == 15 && frac == 8) {"),
    ("e5m2_exponent_bias", "(int)expo - 17", "(int)expo - 16"),
    ("f8_formats_swapped", "    case 1: return oracle_e5m2_to_double(h);", "    case 1: return oracle_e4m3_to_double(h);"),
    ("e2m3_exponent_bias", "(double)(8u + frac) * pow2i((int)expo - 4)", "(double)(8u + frac) * pow2i((int)expo - 3)"),
    ("e3m2_fraction_bits", "    const unsigned frac = h & 0x3u;\n    /* (1 + frac/4) * 2^(expo-3)", "    const unsigned frac = h & 0x1u;\n    /* (1 + frac/4) * 2^(expo-3)"),
    ("e2m1_sign_bit", "    const unsigned sign = (h >> 3) & 1u;\n    const unsigned expo = (h >> 1) & 0x3u;", "    const unsigned sign = (h >> 4) & 1u;\n    const unsigned expo = (h >> 1) & 0x3u;"),
    ("e2m1_subnormal", "(double)frac * pow2i(-1) : (double)(2u + frac)", "(double)frac * pow2i(-2) : (double)(2u + frac)"),
    ("f6_codes_swapped", "    case 3: return oracle_e2m3_to_double(h);", "    case 3: return oracle_e3m2_to_double(h);"),
    ("f8_abs_missing", "        aacc += fabs(p);\n    }\n    *ref = acc;\n    if (absdot)\n        *absdot = aacc;\n}\n\nvoid oracle_gemm_nt_f8",
     "        aacc += p;\n    }\n    *ref = acc;\n    if (absdot)\n        *absdot = aacc;\n}\n\nvoid oracle_gemm_nt_f8"),
    ("mx_block_of_16", "sa_row[k / 32]", "sa_row[k / 16]"),
    ("mx_scale_bias", "return pow2i((int)e - 127);", "return pow2i((int)e - 128);"),
    ("mx_b_scale_dropped", " *\n                         oracle_e8m0_to_double(sb_row[k / 32]);", ";"),
    ("mx_nan_pattern", "    if (e == 255)\n        return NAN;", "    if (e == 254)\n        return NAN;"),
    ("mx_sampled_scale_row", "SA + bidx[s] * sSA + iidx[s] * ldsa", "SA + bidx[s] * sSA + jidx[s] * ldsa"),
    ("mx_batch_scale_stride", "*sa_row = SA + b * sSA + i * ldsa;", "*sa_row = SA + b * sSB + i * ldsa;"),
    ("bf16_sampled_ij_swapped", "iidx[s] * lda, B + bidx[s] * sB + jidx[s] * ldb, K, ref + s,\n",
     "jidx[s] * lda, B + bidx[s] * sB + iidx[s] * ldb, K, ref + s,\n"),
]


@pytest.mark.parametrize("name,orig,planted", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, orig, planted):
    assert SRC.count(orig) >= 1, "mutation site vanished from the oracle source"
    lib = obuild.build_variant(SRC.replace(orig, planted), str(tmp_path), "oracle_" + name)
    orc = oracle.Oracle(lib)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, IndexError, ValueError):
            failed.append(pin.__name__)
    assert failed, "planted mistake %r passed every pin" % name
