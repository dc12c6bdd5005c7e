"""The pins have teeth: each plausible mistake planted in a copy of the oracle
(a dropped term, a wrong sign, an off-by-one level, a wrong bit order or
summation order, a wrong constant) makes the oracle pin suite fail.  The
mutants are compiled from the oracle's source on the CPU and never touch the
CUDA path."""
import concurrent.futures as cf
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "bitscom_oracle.cpp")

MUTANTS = {
    "qmax_off_by_one": ("float qmax = (float)((1 << (bits - 1)) - 1);\n        x = amax / qmax;",
                        "float qmax = (float)((1 << (bits - 1)));\n        x = amax / qmax;"),
    "ef_sign": ("err_out[e] = val - d;", "err_out[e] = d - val;"),
    "ef_add_dropped": ("for (int64_t i = 0; i < n; ++i) v[i] = v[i] + err[i];", ";"),
    "ties_away_from_zero": ("if (frac > 0.5f) return f + 1.0f;", "if (frac >= 0.5f) return f + 1.0f;"),
    "msb_first_packing": ("(bit << (pos % 8))", "(bit << (7 - pos % 8))"),
    "sum_seeded_with_zero": ("acc = (w == 0) ? d : acc + d;", "acc = acc + d;"),
    "reverse_rank_order": ("for (int w = 0; w < W; ++w) {\n            float s = orc_f16_to_f32",
                           "for (int w = W - 1; w >= 0; --w) {\n            float s = orc_f16_to_f32"),
    "philox_multiplier": ("M0 = 0xD2511F53u", "M0 = 0xD2511F55u"),
    "philox_weyl": ("W1 = 0xBB67AE85u", "W1 = 0xBB67AE87u"),
    "sr_flipped": ("(double)f + (double)u < (double)t", "(double)f + (double)u > (double)t"),
    "sr_uniform_from_high_bits": ("float u = (float)(r & 0x7FFFFFu) * (1.0f / 8388608.0f);",
                                  "float u = (float)(r >> 8) * (1.0f / 16777216.0f);"),
    "sr_fraction_rounded": ("(double)f + (double)u < (double)t", "u < t - f"),
    "offset_off_by_one": ("return (uint32_t)(q + (1 << (bits - 1)));", "return (uint32_t)(q + (1 << (bits - 1)) - 1);"),
    "mean_over_block": ("x = sum / (float)n_valid;", "x = sum / (float)B;"),
    "fp16_truncates": ("if (rem > half || (rem == half && (M & 1u))) M += 1;", ";"),
    "no_scale_clamp": ("if (x > 65504.0f) x = 65504.0f;", ";"),
    "left_fold_mean": ("return tree_sum(a, n / 2) + tree_sum(a + n / 2, n / 2);",
                       "float acc = 0.0f; for (int64_t i = 0; i < n; ++i) acc += a[i]; return acc;"),
    "stage2_ef_dropped": ("r[i] = r[i] + err2[i];", "r[i] = r[i];"),
    "bf16_truncates": ("if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) kept += 1;", ";"),
    "mul_inside_product": ("d[i] = s * (float)q;\n    }", "d[i] = s * ((float)q * mul);\n    }"),
    "mul_applied_twice": ("float y = d[i] * mul;", "float y = d[i] * mul * mul;"),
    "fwht_sign": ("x[j + h] = a - b;", "x[j + h] = b - a;"),
    "inverse_without_1_over_H": ("for (int64_t i = 0; i < n; ++i) d[i] = d[i] * inv;", ";"),
    "encoder_skips_rotation": ("if (p->hadamard) orc_fwht(v, n, p->hadamard);", ";"),
    "qwd_reference_not_advanced": ("return orc_qwd_apply(codes, scales, n, p, ref, NULL, 0);", "return 0;"),
    "qwd_difference_sign": ("d[i] = wi - ref[i];", "d[i] = ref[i] - wi;"),
    "local_sum_seeded_with_zero": ("s = (w == 0) ? v : s + v;", "s = s + v;"),
    "local_sum_reverse_order": ("for (int32_t w = 0; w < W; ++w) {\n            float v = (dtype == 0) ? ((const float*)x[w])[i]",
                                "for (int32_t w = W - 1; w >= 0; --w) {\n            float v = (dtype == 0) ? ((const float*)x[w])[i]"),
    "fma_in_feedback": ("float d = s * (float)q;          /* separate roundings, no FMA */\n                err_out[e] = val - d;",
                        "err_out[e] = fmaf(-s, (float)q, val);"),
}


def _run(name, old, new, tmp):
    src = open(SRC).read()
    assert src.count(old) == 1, f"{name}: pattern not found exactly once"
    path = os.path.join(tmp, f"{name}.cpp")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = os.path.join(tmp, f"{name}.so")
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math",
                           "-fPIC", "-shared", "-I", os.path.join(ROOT, "oracle"), path, "-o", lib, "-lm"])
    env = dict(os.environ, BITSCOM_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    return name, r.returncode


def test_every_mutant_fails_a_pin():
    with tempfile.TemporaryDirectory() as tmp:
        with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
            results = list(ex.map(lambda kv: _run(kv[0], *kv[1], tmp), MUTANTS.items()))
    survivors = [n for n, rc in results if rc == 0]
    assert not survivors, f"mutants that pass every pin: {survivors}"
