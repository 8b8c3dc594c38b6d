"""The oracle against facts outside itself (see tests/pins.py), and proof
that the pins have teeth: copies of the oracle with a planted mistake each
fail at least one pin."""
import inspect
import os
import shutil

import numpy as np

import pytest

import pins
from oracle import build as obuild
from oracle import oracle as orc


@pytest.fixture(scope="module")
def lib():
    return orc._load()


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(check, lib):
    check(lib)


# (what goes wrong, text in msa_oracle.c, replacement)
MUTATIONS = [
    ("causal mask off by one", "if (k <= pos && k < seq) keys[nk++] = k;",
     "if (k < pos && k < seq) keys[nk++] = k;"),
    ("query at the head instead of the tail",
     "const int64_t pos = seq - qlen + (t - cu_q[b]);\n        const int P",
     "const int64_t pos = (t - cu_q[b]);\n        const int P"),
    ("V scale dropped", "o[d] += e * (g_dec[row[ORACLE_D + d]] * v_scale);",
     "o[d] += e * (g_dec[row[ORACLE_D + d]]);"),
    ("V read from the K half", "o[d] += e * (g_dec[row[ORACLE_D + d]] * v_scale);",
     "o[d] += e * (g_dec[row[d]] * v_scale);"),
    ("score sign flipped", "s[i] = dot * softmax_scale;",
     "s[i] = -dot * softmax_scale;"),
    ("GQA head map interleaved", "const int hq = h * G + g;",
     "const int hq = g * Hkv + h;"),
    ("repeats counted twice", "if (dup) continue;                                    /* R4 */",
     "(void)dup;"),
    ("lse without the max", "lse[n * Hq + hq] = m + log(sum);",
     "lse[n * Hq + hq] = log(sum);"),
    ("softmax scale dropped", "s[i] = dot * softmax_scale;", "s[i] = dot;"),
    ("CSR keeps the last repeat",
     "for (int i = 0; i < j; ++i)\n                            dup |=",
     "for (int i = j + 1; i < ORACLE_TOPK; ++i)\n                            dup |="),
    ("CSR row offset floors the page count",
     "off[b + 1] = off[b] + (seq + ORACLE_PAGE - 1) / ORACLE_PAGE;\n    }\n    if (off[B] > total_rows)",
     "off[b + 1] = off[b] + seq / ORACLE_PAGE;\n    }\n    if (off[B] > total_rows)"),
    ("CSR keeps future pages", "if (p > own) continue;", "(void)own;"),
    ("combine weights not normalised",
     "const double w = exp(l - L);", "const double w = exp(l - M);"),
    ("E4M3 subnormal exponent", "v = ldexp((double)m, -9);",
     "v = ldexp((double)m, -10);"),
    ("E4M3 encoder rounds ties away from zero",
     "(r > 0.5 || (r == 0.5 && fmod(f, 2.0) == 1.0))", "(r >= 0.5)"),
    ("E4M3 encoder truncates", "(r > 0.5 || (r == 0.5 && fmod(f, 2.0) == 1.0))",
     "(0)"),
    ("E2M1 exponent bias 0", "ldexp(1.0 + 0.5 * m, e - 1)",
     "ldexp(1.0 + 0.5 * m, e)"),
    ("NVFP4 nibble order swapped",
     "(e & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF)",
     "(e & 1) ? (uint8_t)(byte & 0xF) : (uint8_t)(byte >> 4)"),
    ("NVFP4 block of 8 elements", "scales[t * (ORACLE_D / 16) + e / 16]",
     "scales[t * (ORACLE_D / 16) + e / 8 % 8]"),
    ("NVFP4 V slot written over K", "s * ORACLE_D + e] =", "0 * s + e] ="),
    ("BF16 exponent bias 126", "ldexp(1.0 + (double)m / 128.0, e - 127)",
     "ldexp(1.0 + (double)m / 128.0, e - 126)"),
    ("BF16 mantissa read as 6 bits", "ldexp(1.0 + (double)m / 128.0, e - 127)",
     "ldexp(1.0 + (double)(m & 0x3F) / 64.0, e - 127)"),
    ("BF16 query without q_scale",
     "qv[d] = (q16 ? oracle_bf16_decode(q16[at]) : g_dec[q[at]]) * q_scale;",
     "qv[d] = q16 ? oracle_bf16_decode(q16[at]) : g_dec[q[at]] * q_scale;"),
    ("BF16 query of the neighbouring head",
     "const int64_t at = (t * Hq + hq) * ORACLE_D + d;",
     "const int64_t at = (t * Hq + (q16 ? hq ^ 1 : hq)) * ORACLE_D + d;"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new, tmp_path):
    src = open(obuild.SRC).read()
    assert src.count(old) == 1, "mutation anchor not unique: %s" % name
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    libpath = str(tmp_path / "libmutant.so")
    obuild.build_from(str(path), libpath)
    mlib = orc.load_library(libpath)
    caught = []
    for check in pins.ALL_CHECKS:
        try:
            check(mlib)
        except AssertionError:
            caught.append(check.__name__)
        except (ValueError, IndexError):
            caught.append(check.__name__)
    assert caught, "no pin caught: %s" % name


def test_schedule_pins():
    pins.check_schedule()


# (what goes wrong, text in oracle.schedule, replacement)
SCHEDULE_MUTATIONS = [
    ("chunk one token too long", "C = 128 // w.G", "C = 128 // w.G + 1"),
    ("chunks sized by query heads", "C = 128 // w.G", "C = 128 // w.Hq"),
    ("requests outer, KV heads inner",
     "for h in range(w.Hkv):\n        for b in range(w.B):",
     "for b in range(w.B):\n        for h in range(w.Hkv):"),
    ("last short chunk dropped", "for c in range(a, e, C):",
     "for c in range(a, e - C + 1, C):"),
    ("count not clipped at the row end", "min(C, e - c)", "C"),
]


@pytest.mark.parametrize("name,old,new", SCHEDULE_MUTATIONS,
                         ids=[m[0] for m in SCHEDULE_MUTATIONS])
def test_schedule_planted_mistake_is_caught(name, old, new):
    src = inspect.getsource(orc.schedule)
    assert src.count(old) == 1, "mutation anchor not unique: %s" % name
    ns = {"np": np}
    exec(src.replace(old, new), ns)
    with pytest.raises(AssertionError):
        pins.check_schedule(ns["schedule"])
