"""Plants plausible mistakes in a copy of the oracle and checks the pins catch each.

Every mutant is compiled from the oracle's own C source with one edit; the pin
suite is then run against it in a subprocess and must fail.  CPU only.
"""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "csa_oracle.c")

MUTANTS = {
    "relu dropped": ("acc += w[h] * (dot > 0.0 ? dot : 0.0);", "acc += w[h] * dot;"),
    "w index off by one": ("acc += w[h] * (dot > 0.0 ? dot : 0.0);",
                           "acc += w[(h + 1) % Hi] * (dot > 0.0 ? dot : 0.0);"),
    "tie to higher index": ("return (x->j < y->j) ? -1 : (x->j > y->j);",
                            "return (x->j > y->j) ? -1 : (x->j < y->j);"),
    "ascending sort": ("if (x->key > y->key) return -1;\n    if (x->key < y->key) return 1;",
                       "if (x->key < y->key) return -1;\n    if (x->key > y->key) return 1;"),
    "rope sign": ("x[2 * i] = x0 * c + x1 * s;", "x[2 * i] = x0 * c - x1 * s;"),
    "rope frequency": ("pow(base, -2.0 * (double)i / (double)R)", "pow(base, -1.0 * (double)i / (double)R)"),
    "rope on first dims": ("double *x = o + (int64_t)h * V + (V - R);", "double *x = o + (int64_t)h * V;"),
    "window off by one": ("for (int32_t r = pos - nwin + 1; r <= pos; ++r, ++u)",
                          "for (int32_t r = pos - nwin; r < pos; ++r, ++u)"),
    "visibility off by one": ("const int32_t vis = (pos + 1) / c->ratio;\n    const int32_t nwin",
                              "const int32_t vis = pos / c->ratio;\n    const int32_t nwin"),
    # (vis >= K in place of vis > K is an equivalent mutant: scoring then keeps all K rows)
    "bypass too wide": ("if (vis > K || (flags & ORC_FORCE_SCORE))", "if (vis > 2 * K || (flags & ORC_FORCE_SCORE))"),
    "values from rope dims": ("oh[v] += p * rows[(int64_t)u * D + v];",
                              "oh[v] += p * rows[(int64_t)u * D + (D - V) + v];"),
    "no max subtraction scale": ("s[u] = scale * dot;", "s[u] = dot;"),
    "dropped hca": ("for (int32_t r = 0; r < vis2; ++r, ++u)", "for (int32_t r = 0; r < 0; ++r, ++u)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {name}"
    with tempfile.TemporaryDirectory() as td:
        c = os.path.join(td, "m.c")
        so = os.path.join(td, "m.so")
        open(c, "w").write(src.replace(old, new, 1))
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", so, c, "-lm"],
                       check=True)
        env = dict(os.environ, CSA_ORACLE_LIB=so)
        r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                            os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                           env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
        assert r.returncode != 0, f"pins did not catch mutant '{name}'"
