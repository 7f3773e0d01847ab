"""The oracle's pins must catch plausible mistakes.

Each mutant below is a copy of the oracle's C source with one deliberate error
(a wrong rounding rule, a fused reconstruction, zero padding, a dropped term, a
wrong index ...). The mutant is compiled on the CPU into a temporary library and
the pin suite (tests/test_oracle.py) is run against it in a subprocess; the
suite must fail for every mutant."""
import concurrent.futures as cf
import os
import subprocess
import sys
import tempfile

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "kivi_oracle.c")

MUTANTS = {
    "round_half_away": ("float r = rintf(t);", "float r = roundf(t);"),
    "fused_recon": ("float prod = (float)q * s;\n    float out = prod + z;",
                    "float prod = 0.0f; (void)prod;\n    float out = fmaf((float)q, s, z);"),
    "zero_padding": ("buf[i] = real[n_real - 1];", "buf[i] = 0.0f;"),
    "no_signed_zero_fix": ("mn = mn + 0.0f;", ";"),
    "no_signed_zero_fix_max": ("mx = mx + 0.0f;", ";"),
    "reciprocal_multiply": ("float t = a / s;", "float t = a * (1.0f / s);"),
    "pack_high_bits_first": ("(bit % 8)", "(8 - bits - bit % 8)"),
    "key_meta_ignores_s_off": ("((long)bh * ng_cap + (s_off / G + g)) * D + d",
                               "((long)bh * ng_cap + g) * D + d"),
    "value_meta_ignores_s_off": ("((long)bh * s_cap + s_off + t) * ngd + j",
                                 "((long)bh * s_cap + t) * ngd + j"),
    "head_stride_from_n_flush": ("xb = x + (long)bh * x_bh_stride * D;\n        for (int g",
                                 "xb = x + (long)bh * n_flush * D;\n        for (int g"),
    "flush_trigger_off_by_one": ("if (over < group_size)", "if (over <= group_size)"),
    "half_exponent_bias": ("ldexpf((float)(1024 + m), e - 25)", "ldexpf((float)(1024 + m), e - 24)"),
    "half_round_ties_away": ("double n = rint(a / ldexp(1.0, E - 10));",
                             "double n = floor(a / ldexp(1.0, E - 10) + 0.5);"),
    "dropped_sm_scale": ("score[t] = sm_scale * acc;", "score[t] = acc;"),
    "values_read_as_keys": ("V[(long)t * D + d] = (double)vf[(long)t * D + d];",
                            "V[(long)t * D + d] = (double)kf[(long)t * D + d];"),
    "missing_normalisation": ("oh[d] = T > 0 ? acc / denom : 0.0;", "oh[d] = acc;"),
    "f16_scale_codes_use_fp32_scale": ("        s = orc_half_to_float(orc_float_to_half(s)); /* the stored binary16 scale */",
                                       "        ;"),
    "f16_scale_read_as_fp32": ("        return orc_half_to_float(((const uint16_t*)scale)[m]);",
                               "        return ((const float*)scale)[m];"),
    "f16_scale_head_stride_of_fp32": ("long esz = (bits & ORC_SCALE_F16) ? 2 : 4;", "long esz = 4;"),
    "gqa_modulo_mapping": ("const uint16_t* qh = q + ((long)b * Hq + h) * D;",
                           "const uint16_t* qh = q + ((long)b * Hq + (h % group) * Hkv + hk) * D;"),
}


def _run_mutant(name, old, new, tmp):
    src = open(SRC).read()
    assert src.count(old) >= 1, name
    mut = os.path.join(tmp, name + ".c")
    with open(mut, "w") as f:
        f.write(src.replace(old, new))
    lib = os.path.join(tmp, name + ".so")
    subprocess.run(["gcc", *oracle.CFLAGS, "-I", os.path.join(ROOT, "oracle"), "-o", lib, mut, "-lm"],
                   check=True)
    env = dict(os.environ, KIVI_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return name, r.returncode


def test_every_mutant_is_caught():
    with tempfile.TemporaryDirectory() as tmp:
        with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
            futs = [ex.submit(_run_mutant, n, o, w, tmp) for n, (o, w) in MUTANTS.items()]
            results = dict(f.result() for f in futs)
    survivors = [n for n, rc in results.items() if rc == 0]
    assert not survivors, "mutants not caught by the oracle pins: %s" % survivors
