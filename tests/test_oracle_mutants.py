"""The oracle's pins catch plausible mistakes: each case plants one mistake in a copy of the
oracle's C source (a wrong shift or zero point, a flipped sign, a codec bias, a tie rule, a
transposed or dropped GEMV term ...), builds it the way the oracle is built, and runs the pin
tests (tests/test_oracle_*.py) against that build in a child process. Every mutant must make
at least one pin fail; the unmodified source, built the same way, must pass them all.

Mistakes are planted on the CPU only, in a temporary copy; the oracle itself is untouched.
"""
import concurrent.futures
import os
import re
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE = os.path.join(ROOT, "oracle")
PINS = ["tests/test_oracle_codecs.py", "tests/test_oracle_pn.py", "tests/test_oracle_quantizer.py",
        "tests/test_oracle_gemv_nvfp4.py"]

# name, text to replace, replacement, occurrences to replace (0 = all; the text must occur)
MUTANTS = [
    ("layout_element_index_shift_everywhere", "p->bits * (t >> 1) + 16 * (t & 1)", "p->bits * t", 0),
    ("decode_halves_swapped", "int shift = p->bits * (t >> 1) + 16 * (t & 1);\n    return",
     "int shift = p->bits * (t >> 1) + 16 * ((t & 1) ^ 1);\n    return", 1),
    ("pn3t_zero_point_3", "p->cpw = 10; p->z = 4;", "p->cpw = 10; p->z = 3;", 1),
    ("pn4t_zero_point_7", "p->cpw = 8;  p->z = 8;", "p->cpw = 8;  p->z = 7;", 1),
    ("decode_sign_flipped", "out[r * K + b * p.blk + e] = (float)(d * (double)(n - p.z));\n            }\n        }\n    }",
     "out[r * K + b * p.blk + e] = (float)(d * (double)(p.z - n));\n            }\n        }\n    }", 1),
    ("decode_d_from_second_byte", "double d = pnq_ref_fp16_to_double(rd16(block));\n            for (int e = 0; e < p.blk; ++e) {\n                int n",
     "double d = pnq_ref_fp16_to_double(rd16(block + 1));\n            for (int e = 0; e < p.blk; ++e) {\n                int n", 1),
    ("fp16_subnormal_scale", "v = ldexp((double)f, -24);", "v = ldexp((double)f, -23);", 1),
    ("fp16_exponent_bias", "v = ldexp(1024.0 + (double)f, e - 25);", "v = ldexp(1024.0 + (double)f, e - 24);", 1),
    ("fp16_encode_ties_away", "double r = nearbyint(q);", "double r = round(q);", 1),
    ("bf16_wrong_half", "uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;", 1),
    ("e2m1_subnormal_step", "(e == 0) ? 0.5 * m :", "(e == 0) ? 1.0 * m :", 1),
    ("e4m3_bias_8", "v = ldexp(1.0 + m / 8.0, e - 7);", "v = ldexp(1.0 + m / 8.0, e - 8);", 1),
    ("e4m3_max_is_nan_missing", "else if (e == 15 && m == 7)\n        v = NAN;", "else if (0)\n        v = NAN;", 1),
    ("quantizer_tie_to_smaller_m", "if (!found || err <= best) {", "if (!found || err < best) {", 1),
    ("quantizer_sigma_flipped", "(fabs(mn) > mx) ? 1.0 : -1.0", "(fabs(mn) > mx) ? -1.0 : 1.0", 1),
    ("quantizer_m_grid", "double m = (50.0 + 2.0 * i) / 100.0;", "double m = (50.0 + 2.0 * i) / 101.0;", 1),
    ("quantizer_fewer_candidates", "for (int i = 0; i < 36; ++i) {", "for (int i = 0; i < 35; ++i) {", 1),
    ("quantizer_clamp_high", "if (q > (double)(2 * p->z - 1)) q = (double)(2 * p->z - 1);",
     "if (q > (double)(2 * p->z)) q = (double)(2 * p->z);", 1),
    ("quantizer_zero_group_d_negative", "uint16_t dbits = 0x0000;", "uint16_t dbits = 0x8000;", 1),
    ("validate_inf_not_flagged", "if (!isfinite(d)) bad = 1;", "if (isnan(d)) bad = 1;", 1),
    ("validate_bit31_ignored", "if ((w >> 31) & 1) bad = 1;", "", 1),
    ("validate_pn4t_reserved_bits", "if (type == PNQ_REF_PN3T)\n                for (int i = 0; i < 8; ++i) {",
     "if (1)\n                for (int i = 0; i < 8; ++i) {", 1),
    ("nvfp4_nibbles_swapped", "(k & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF)",
     "(k & 1) ? (uint8_t)(byte & 0xF) : (uint8_t)(byte >> 4)", 1),
    ("nvfp4_scale_per_32", "scales_row[k / 16]", "scales_row[k / 32]", 1),
    ("nvfp4_global_dropped", "return pnq_ref_e2m1_to_double(c) * s * (double)g;",
     "return pnq_ref_e2m1_to_double(c) * s;", 1),
    ("nvfp4_validate_negative_zero_accepted", "if (s & 0x80) bad = 1;", "if ((s & 0x80) && (s & 0x7F)) bad = 1;", 1),
    ("nvfp4_validate_global_zero_accepted", "int g_ok = isfinite(g) && g > 0.0f;", "int g_ok = isfinite(g) && g >= 0.0f;", 1),
    ("gemv_x_transposed", "double t = (double)wrow[k] * xd[(int64_t)m * K + k];",
     "double t = (double)wrow[k] * xd[(int64_t)k * M + m];", 1),
    ("gemv_last_term_dropped", "for (int64_t k = 0; k < K; ++k) {\n            double t = (double)wrow[k]",
     "for (int64_t k = 0; k + 1 < K; ++k) {\n            double t = (double)wrow[k]", 1),
    ("gemv_abs_sum_signed", "a += fabs(t);\n        }\n        Y[(int64_t)m * N + n] = s;",
     "a += t;\n        }\n        Y[(int64_t)m * N + n] = s;", 1),
    ("gemv_nvfp4_rows_swapped", "nvfp4_weight(codes + n * (K / 2), scales + n * (K / 16), g, k) *",
     "nvfp4_weight(codes + (N - 1 - n) * (K / 2), scales + (N - 1 - n) * (K / 16), g, k) *", 1),
]


def build_variant(dirpath, old=None, new=None, count=0):
    src = open(os.path.join(ORACLE, "pnq_oracle.c")).read()
    if old is not None:
        assert old in src, "the mutated text is no longer in the oracle source"
        src = src.replace(old, new, count if count else -1)
    d = os.path.join(dirpath, "src")
    os.makedirs(d)
    with open(os.path.join(d, "pnq_oracle.c"), "w") as f:
        f.write(src)
    shutil.copy(os.path.join(ORACLE, "pnq_oracle.h"), os.path.join(d, "pnq_oracle.h"))
    so = os.path.join(dirpath, "libpnq_oracle_variant.so")
    # the flags of oracle.build()
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fno-fast-math", "-ffp-contract=off", "-shared", "-fPIC",
                           os.path.join(d, "pnq_oracle.c"), "-o", so, "-lm"])
    return so


def run_pins(so, exitfirst=True):
    env = dict(os.environ, PNQ_ORACLE_LIB=so)
    cmd = [sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", "-m", "not gpu"]
    if exitfirst:
        cmd.append("-x")
    return subprocess.run(cmd + PINS, env=env, capture_output=True, text=True, timeout=600, cwd=ROOT)


@pytest.fixture(scope="module")
def mutant_runs(tmp_path_factory):
    """Every mutant built and run against the pins, several child processes at a time."""
    def one(m):
        name, old, new, count = m
        return name, run_pins(build_variant(str(tmp_path_factory.mktemp(name)), old, new, count))
    workers = max(1, min(8, len(os.sched_getaffinity(0))))
    with concurrent.futures.ThreadPoolExecutor(workers) as ex:
        return dict(ex.map(one, MUTANTS))


def test_unmodified_source_passes_the_pins(tmp_path):
    r = run_pins(build_variant(str(tmp_path)), exitfirst=False)
    assert r.returncode == 0, r.stdout[-3000:]


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_pins_reject_planted_mistake(mutant_runs, name):
    r = mutant_runs[name]
    failed = re.findall(r"^(?:FAILED|ERROR) (\S+)", r.stdout, flags=re.M)
    assert r.returncode == 1 and failed, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
