"""Every pin battery must catch a planted mistake in the oracle.

Each case copies the oracle's C source, changes one expression (a sign, an
index, a dropped term, a transposed operand), compiles the copy on the CPU and
runs the pin checks against it; at least one check must fail.  The real oracle
is never modified.
"""
import os

import pytest

import oracle
import oracle_checks as oc

MUTANTS = [
    ("rope sign", "y[i] = x1 * c - x2 * s;", "y[i] = x1 * c + x2 * s;"),
    ("rope partner index", "double x1 = x[i], x2 = x[i + half];",
     "double x1 = x[i], x2 = x[(i + 1) % half + half];"),
    ("rope pass-through dropped", "        y[j] = x[j];", "        y[j] = 0.0;"),
    ("rope frequency exponent", "(double)(2 * i) / (double)rotary_dim", "(double)(i) / (double)rotary_dim"),
    ("rope angle fp32 table skipped", "cos_half[i] = (float)cos(ang);", "cos_half[i] = (float)cos(ang + 1e-3);"),
    ("score scale", "double scale = 1.0 / sqrt((double)head_dim);", "double scale = 1.0 / (double)head_dim;"),
    ("softmax normaliser", "double w = s[j] / z;", "double w = s[j];"),
    ("lse drops the max", "*lse = m + log(z);", "*lse = log(z);"),
    ("sink sign", "exp(sink - *lse)", "exp(*lse - sink)"),
    ("sink applied twice", "out[d] *= f;", "out[d] *= f * f;"),
    ("gqa mapping transposed", "const int h = kv * g + hh;", "const int h = hh * Hkv + kv;"),
    ("value row is the key", "load_cached_row(L, vnew_bits, 0, vs, vals + n * D);",
     "load_cached_row(L, knew_bits, 0, vs, vals + n * D);"),
    ("new key not rotated", "(const void *)kq : (const void *)kb;", "(const void *)kq : (const void *)kin;"),
    ("ring slot off by one", "slot = c % (L->window - 1);", "slot = (c + 1) % (L->window - 1);"),
    ("roll keeps the oldest", "first = 1; /*", "first = 0; /*"),
    ("roll never shifts", "if (c >= L->window) {", "if (c > 1000000000) {"),
    ("bf16 truncates", "double r = rint(ldexp(a, 7 - E));", "double r = floor(ldexp(a, 7 - E));"),
    ("bf16 exponent", "int E = e - 1;           /* a = (2m)", "int E = e;           /* a = (2m)"),
    ("full cache keeps one less", "if (layer_type != ORC_SLIDING)\n        return context;",
     "if (layer_type != ORC_SLIDING)\n        return context > 0 ? context - 1 : 0;"),
    ("footprint counts K only", "int64_t per_entry = 2LL *", "int64_t per_entry = 1LL *"),
    ("gate sign", "exp(-(double)gate[", "exp((double)gate["),
    ("e4m3 exponent bias", "ldexp((double)(8 + m), e - 10)", "ldexp((double)(8 + m), e - 9)"),
    ("e4m3 subnormal quantum", "ldexp((double)m, -9)", "ldexp((double)m, -8)"),
    ("e4m3 overflow to NaN", "if (v > 448.0)\n        return sign | 0x7E;", "if (v > 448.0)\n        return sign | 0x7F;"),
    ("e4m3 ties away from zero", "double v = ldexp(rint(ldexp(a, 3 - E)), E - 3);",
     "double v = ldexp(round(ldexp(a, 3 - E)), E - 3);"),
    ("fp8 quantise multiplies by the scale", "orc_f64_to_e4m3(knew[d] / ks)", "orc_f64_to_e4m3(knew[d] * ks)"),
    ("fp8 value scale dropped", "load_cached_row(L, vc, j, vs, vals + n * D);",
     "load_cached_row(L, vc, j, 1.0, vals + n * D);"),
    ("roll shift in elements, not bytes", "memmove(kc, kc + D * esize,", "memmove(kc, kc + D,"),
    ("tokens share one position", "ctx[b] = context[b] + t;", "ctx[b] = context[b];"),
    ("tokens read the wrong q", "q + ((size_t)b * T + t) * Hq * D", "q + ((size_t)b * T) * Hq * D"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new):
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = oracle.build(str(path), str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(lib)
    failed = []
    for check in oc.ALL_CHECKS:
        try:
            check(orc)
        except (AssertionError, ValueError, FloatingPointError) as e:
            failed.append(check.__name__)
    assert failed, f"no pin caught the mutant {name!r}"
