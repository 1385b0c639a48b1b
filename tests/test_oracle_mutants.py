"""The pins catch mistakes planted in the oracle.

Each case copies oracle.c, plants one plausible mistake (a dropped term, a
wrong stride or index, a transposed operand, a wrong sign, a misplaced
remainder, a missing wrap, an accum folded twice), builds the mutant and runs
tests/test_oracle_pins.py against it in a subprocess (ORACLE_LIB points the
oracle package at the mutant).  The pin suite must fail for every mutant,
and pass for an unmodified copy built the same way."""
import os
import subprocess
import sys

import pytest

from conftest import ROOT

SRC = os.path.join(ROOT, "oracle", "oracle.c")
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

MUTANTS = {
    "full sum drops the last element": ("s += (double)x[i];\n        a += fabs((double)x[i]);\n    }\n    *sum = s;",
                                        "if (i + 1 < n) s += (double)x[i];\n        a += fabs((double)x[i]);\n    }\n    *sum = s;"),
    "full max keeps the first element": ("        if (x[i] > m)\n            m = x[i];\n    *out = m;",
                                         "        if (x[i] > m && 0)\n            m = x[i];\n    *out = m;"),
    "dense rows use a wrong stride": ("out[r] = seg_sum(x + r * len, len, init, &abs_out[r], ainit);",
                                      "out[r] = seg_sum(x + r * (len - (len > 1)), len, init, &abs_out[r], ainit);"),
    "ragged rows read one element short": ("out[r] = seg_sum(x + off[r], off[r + 1] - off[r], init, &abs_out[r], ainit);",
                                           "out[r] = seg_sum(x + off[r], off[r + 1] - off[r] - (off[r + 1] > off[r]), init, &abs_out[r], ainit);"),
    "accum folds the old value twice": ("double init = accum ? (double)dst_old[r] : 0.0;\n        double ainit = accum ? fabs((double)dst_old[r]) : 0.0;\n        out[r] = seg_sum(x + r * len",
                                        "double init = accum ? 2.0 * (double)dst_old[r] : 0.0;\n        double ainit = accum ? fabs((double)dst_old[r]) : 0.0;\n        out[r] = seg_sum(x + r * len"),
    "colprod is transposed": ("p *= (double)x[i * C + j];", "p *= (double)x[(i * C + j) % R * C + (i * C + j) / R % C];"),
    "int32 colprod saturates instead of wrapping": ("p *= (uint32_t)x[i * C + j];",
                                                    "p = (uint64_t)p * (uint32_t)x[i * C + j] > 0xffffffffu ? 0xffffffffu : p * (uint32_t)x[i * C + j];"),
    "thread fold puts the remainder in slot 0": ("s[i - c] = s[i - c] + a[i];", "s[0] = s[0] + a[i];"),
    "thread fold collapses in a different order": ("    s[0] = s[0] + s[2];\n    s[1] = s[1] + s[3];",
                                                   "    s[0] = s[0] + s[1];\n    s[1] = s[2] + s[3];"),
    "thread fold pairs the upper half differently": ("    s[4] = s[4] + s[6];\n    s[5] = s[5] + s[7];",
                                                      "    s[4] = s[4] + s[5];\n    s[5] = s[6] + s[7];"),
    "thread fold's second collapse pairs differently": ("    s[0] = s[0] + s[4];\n    s[1] = s[1] + s[5];\n    return s[0] + s[1];",
                                                        "    s[0] = s[0] + s[1];\n    s[4] = s[4] + s[5];\n    return s[0] + s[4];"),
    "int16 column sum does not wrap": ("            w &= mask;\n            if (is_signed && (w >> (bits - 1)) & 1u)\n                m = (int64_t)w - (int64_t)(mask + 1);",
                                       "            if (0 && is_signed && (w >> (bits - 1)) & 1u)\n                m = (int64_t)w - (int64_t)(mask + 1);"),
    "bf16 decode shifts one bit short": ("const uint32_t w = (uint32_t)b << 16;", "const uint32_t w = (uint32_t)b << 15;"),
    "uint16 elements read as signed": ("    default: return (int64_t)((const uint16_t *)x)[k];",
                                       "    default: return (int64_t)((const int16_t *)x)[k];"),
    "uint32 elements read as signed": ("case ORC_U32: return (int64_t)((const uint32_t *)x)[k];",
                                       "case ORC_U32: return (int64_t)((const int32_t *)x)[k];"),
    "column max compares the wrong way": ("                acc = v > acc ? v : acc;\n            else\n                acc = v < acc ? v : acc;\n        }\n        out[j] = acc;",
                                          "                acc = v < acc ? v : acc;\n            else\n                acc = v < acc ? v : acc;\n        }\n        out[j] = acc;"),
    "empty ragged row's max starts from 0": ("float init = accum ? dst_old[r] : -INFINITY;", "float init = accum ? dst_old[r] : 0.0f;"),
    "dense rows max ignores accum": ("if (accum && dst_old[r] > m)", "if (0 && accum && dst_old[r] > m)"),
    "typed float rows ignore accum": ("        if (accum) {\n            acc = elem_f(dst_old, dtype, r);",
                                      "        if (0) {\n            acc = elem_f(dst_old, dtype, r);"),
    "typed integer rows ignore accum": ("        if (accum) {\n            m = elem_i(dst_old, dtype, r);",
                                        "        if (0) {\n            m = elem_i(dst_old, dtype, r);"),
    "typed integer rows skip the first element": ("            m = elem_i(x, dtype, r * len);\n            k = 1;",
                                                  "            m = elem_i(x, dtype, r * len);\n            k = 2;"),
    "decreasing ragged offsets accepted": ("        if (off[r + 1] < off[r])\n            return ORC_EINVAL;",
                                           "        if (0)\n            return ORC_EINVAL;"),
    "full min keeps the first element": ("        if (x[i] < m)\n            m = x[i];\n    *out = m;",
                                         "        if (x[i] < m && 0)\n            m = x[i];\n    *out = m;"),
    "column fold drops the last row": ("        for (int64_t i = 1; i < R; ++i) {\n            const double v = elem_f(x, dtype, i * C + j);",
                                       "        for (int64_t i = 1; i < R - 1; ++i) {\n            const double v = elem_f(x, dtype, i * C + j);"),
    "full sum|x| forgets the absolute value": ("        a += fabs((double)x[i]);\n    }\n    *sum = s;",
                                               "        a += (double)x[i];\n    }\n    *sum = s;"),
    "empty typed product row starts from 0": ("acc = op == ORC_PROD ? 1.0 : 0.0;", "acc = 0.0;"),
    "half subnormals decoded with a wrong scale": ("v = ldexp((double)f, -24);", "v = ldexp((double)f, -25);"),
    "short thread fold adds accum last": ("        float r = a[0];\n        if (accum)\n            r = r + dst;\n        for (int64_t i = 1; i < n; ++i)\n            r = r + a[i];\n        return r;",
                                          "        float r = a[0];\n        for (int64_t i = 1; i < n; ++i)\n            r = r + a[i];\n        if (accum)\n            r = r + dst;\n        return r;"),
    "half decode uses a wrong exponent bias": ("v = ldexp((double)(f | 0x400), e - 25);", "v = ldexp((double)(f | 0x400), e - 24);"),
}


def _build(tmp_path, name, text):
    src = tmp_path / f"{name}.c"
    lib = tmp_path / f"lib{name}.so"
    src.write_text(text)
    subprocess.run(["gcc", "-std=c99", "-O2", "-fno-fast-math", "-fPIC", "-shared", "-o", str(lib), str(src), "-lm"],
                   check=True)
    return str(lib)


def _run_pins(lib):
    env = dict(os.environ, ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode


def test_unmodified_copy_passes(tmp_path):
    assert _run_pins(_build(tmp_path, "orig", open(SRC).read())) == 0


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation site not found: {name}"
    mutant = text.replace(old, new, 1)
    assert _run_pins(_build(tmp_path, "mutant", mutant)) != 0, f"pins did not catch: {name}"
