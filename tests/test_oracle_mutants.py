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
PINS = ["tests/test_oracle_codecs.py", "tests/test_oracle_gemm.py"]

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
        "out[r * K + k] = dec_fp8(fmt, X[r * K + k]) * dtc_oracle_dec_e8m0(sf[r * kb + k / block]);",
        "out[r * K + k] = dec_fp8(fmt, X[r * K + k]) * dtc_oracle_dec_e8m0(sf[r * kb]);",
    ),
    "b_scaled_with_a_scales": (
        "double* bt = decode_scaled(fmt_b, block, B, sfB, N, K);",
        "double* bt = decode_scaled(fmt_b, block, B, sfA, N, K);",
    ),
    "e5m2_bias_off_by_one": (
        "v = ldexp((double)(4 + m), e - 17); /* (1 + m/4) * 2^(e-15) */",
        "v = ldexp((double)(4 + m), e - 16); /* (1 + m/4) * 2^(e-15) */",
    ),
    "b_decoded_with_a_format": (
        "double* bt = decode_scaled(fmt_b, block, B, sfB, N, K);",
        "double* bt = decode_scaled(fmt_a, block, B, sfB, N, K);",
    ),
    "scale_block_fixed_at_128": (
        "int64_t kb = (K + block - 1) / block;\n    double* out",
        "block = 128;\n    int64_t kb = (K + block - 1) / block;\n    double* out",
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
