"""The oracle's pins must catch plausible mistakes (CPU only).

Each case copies the oracle's C source, plants one mistake (a transposed operand, a dropped term,
a wrong sign, index, bias or rounding rule, a swapped scale), builds the copy with gcc into a
temporary directory and runs the pin suites against it in a subprocess. The suite must fail.
Nothing here touches a GPU.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "dtc_oracle.c")
PINS = ["tests/test_oracle_codecs.py", "tests/test_oracle_gemm.py", "tests/test_oracle_formats.py",
        "tests/test_oracle_sparse.py"]

MUTANTS = {
    "nn_operand_read_as_nt": (
        "bt[n * K + k] = dec16(dtype, b_is_kn(layout) ? B[k * N + n] : B[n * K + k]);",
        "bt[n * K + k] = dec16(dtype, B[n * K + k]);",
    ),
    "transposed_a_read_untransposed": (
        "a[m * K + k] = dec16(dtype, a_is_km(layout) ? A[k * M + m] : A[m * K + k]);",
        "a[m * K + k] = dec16(dtype, A[m * K + k]);",
    ),
    "tt_b_read_as_kn": (
        "static int b_is_kn(int layout) { return layout == DTC_ORACLE_NN || layout == DTC_ORACLE_TN; }",
        "static int b_is_kn(int layout) { return layout != DTC_ORACLE_NT; }",
    ),
    "last_k_term_dropped": (
        "for (int64_t k = 0; k < j->K; ++k) acc += arow[k] * brow[k];",
        "for (int64_t k = 0; k + 1 < j->K; ++k) acc += arow[k] * brow[k];",
    ),
    "f16_sign_lost": (
        "v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */\n    }\n    return sign ? -v : v;",
        "v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */\n    }\n    return v;",
    ),
    "ties_away_from_zero": ("double r = nearbyint(scaled);", "double r = round(scaled);"),
    "truncating_round": ("double r = nearbyint(scaled);", "double r = trunc(scaled);"),
    "bf16_double_rounding_through_float": (
        "round_to_format(x, 8, -126,",
        "round_to_format((double)(float)x, 8, -126,",
    ),
    "e4m3_bias_off_by_one": (
        "v = ldexp((double)(8 + m), e - 10);",
        "v = ldexp((double)(8 + m), e - 9);",
    ),
    "scale_block_index_wrong": (
        "dec_scale(sf_kind, sf[r * kb + k / block]);",
        "dec_scale(sf_kind, sf[r * kb]);",
    ),
    "b_scaled_with_a_scales": (
        "double* bt = decode_scaled(fmt_b, sf_kind, block, B, sfB, N, K);",
        "double* bt = decode_scaled(fmt_b, sf_kind, block, B, sfA, N, K);",
    ),
    "e5m2_bias_off_by_one": (
        "v = ldexp((double)(4 + m), e - 17); /* (1 + m/4) * 2^(e-15) */",
        "v = ldexp((double)(4 + m), e - 16); /* (1 + m/4) * 2^(e-15) */",
    ),
    "b_decoded_with_a_format": (
        "double* bt = decode_scaled(fmt_b, sf_kind, block, B, sfB, N, K);",
        "double* bt = decode_scaled(fmt_a, sf_kind, block, B, sfB, N, K);",
    ),
    "scale_block_fixed_at_128": (
        "int64_t kb = (K + block - 1) / block;\n    int64_t rb = row_bytes(fmt, K);",
        "block = 128;\n    int64_t kb = (K + block - 1) / block;\n    int64_t rb = row_bytes(fmt, K);",
    ),
    "fp4_nibbles_swapped": (
        "int shift = (int)(bit % 8);",
        "int shift = bits == 4 ? 4 - (int)(bit % 8) : (int)(bit % 8);",
    ),
    "fp6_field_read_from_one_byte": (
        "if (shift + bits > 8) v |= (unsigned)row[byte + 1] << 8; /* the field spans two bytes */",
        "",
    ),
    "e2m3_bias_off_by_one": (
        ": ldexp((double)(8 + m), e - 4);  /* (1 + m/8) * 2^(e-1) */",
        ": ldexp((double)(8 + m), e - 3);  /* (1 + m/8) * 2^(e-1) */",
    ),
    "e3m2_subnormal_scale_wrong": (
        "double v = e == 0 ? ldexp((double)m, -4)            /* subnormal: m/4 * 2^(1-3) */",
        "double v = e == 0 ? ldexp((double)m, -3)            /* subnormal: m/4 * 2^(1-3) */",
    ),
    "e2m1_mantissa_ignored": (
        ": ldexp((double)(2 + m), e - 2);  /* (1 + m/2) * 2^(e-1) */",
        ": ldexp(2.0, e - 2);  /* (1 + m/2) * 2^(e-1) */",
    ),
    "ue4m3_sign_not_rejected": ("if (b & 0x80) return NAN;\n", ""),
    "sparse_nn_operand_read_as_nt": (
        "const uint16_t code = b_is_kn(layout) ? B[k * N + n] : B[n * K + k]; /* Bop[k][n] */",
        "const uint16_t code = B[n * K + k]; /* Bop[k][n] */",
    ),
    "sparse_position_fields_swapped": (
        "return (nib >> (2 * j)) & 0x3;",
        "return (nib >> (2 * (1 - j))) & 0x3;",
    ),
    "sparse_nibbles_swapped": (
        "uint8_t nib = (uint8_t)((meta_row[g / 2] >> (4 * (g % 2))) & 0xf);",
        "uint8_t nib = (uint8_t)((meta_row[g / 2] >> (4 * (1 - g % 2))) & 0xf);",
    ),
    "sparse_value_index_wrong": (
        "dec16(dtype, vals[m * (K / 2) + 2 * g + j]);",
        "dec16(dtype, vals[m * (K / 2) + g + j]);",
    ),
    "nvfp4_scales_read_as_e8m0": (
        "return sf_kind == DTC_ORACLE_SF_UE4M3 ? dtc_oracle_dec_ue4m3(c) : dtc_oracle_dec_e8m0(c);",
        "return dtc_oracle_dec_e8m0(c);",
    ),
    "f16_subnormal_scale_wrong": (
        "v = ldexp((double)m, -24); /* subnormal: m * 2^-10 * 2^-14 */",
        "v = ldexp((double)m, -25); /* subnormal: m * 2^-10 * 2^-14 */",
    ),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, "mutation anchor must match the oracle source exactly once"
    mutated = tmp_path / "dtc_oracle_mutant.c"
    mutated.write_text(src.replace(before, after))
    lib = tmp_path / "libdtc_oracle_mutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           "-ffp-contract=off", "-o", str(lib), str(mutated), "-lm"])
    env = dict(os.environ, DTC_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "-m", "not gpu", *PINS], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode != 0, f"planted mistake '{name}' passed every pin:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout
