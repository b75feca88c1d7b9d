"""Plant plausible mistakes in copies of oracle.c and check that the pin suite
catches every one of them (the oracle is pinned to facts, not to itself)."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

# (name, original text, mutated text, replace every occurrence?)
MUTANTS = [
    ("rope sin sign", "r[i] = x1 * c - x2 * s;", "r[i] = x1 * c + x2 * s;", False),
    ("rope frequency exponent", "pow(base, -2.0 * (double)i / (double)d)", "pow(base, -1.0 * (double)i / (double)d)", False),
    ("rope partner index", "double x1 = r[i], x2 = r[i + half];", "double x1 = r[i], x2 = r[(i + 1) % d];", False),
    ("gqa head map", "int g = h / G;", "int g = h % hkv;", False),
    ("dropped scale", "s *= scale;", "s *= 1.0;", False),
    ("strict causal mask", "kpos[j] > qp", "kpos[j] >= qp", True),
    ("lse without max", "*lse = M + log(L);", "*lse = log(L);", False),
    ("values replaced by keys", "const double *vr = vb + j * kstride;", "const double *vr = kb + j * kstride;", False),
    ("merge weight vs max", "double w = exp(l - L);", "double w = exp(l - mx);", False),
    ("decode query position", "ctx, ctx - 1, 1, d,", "ctx, ctx - 2, 1, d,", False),
    ("page slot index", "(j % page)) * (int64_t)d;", "(j / page)) * (int64_t)d;", False),
    ("bf16 ulp", "int q = e - 8;", "int q = e - 9;", False),
    ("append row of head", "double *kd = k_cache + ((int64_t)h * rows + s) * d;",
     "double *kd = k_cache + ((int64_t)s * heads + h) * d;", False),
    ("int8 scale of the wrong token", "(double)scales[r];", "(double)scales[r > 0 ? r - 1 : r];", False),
    ("int8 scale over 128", "float s = amax / 127.0f;", "float s = amax / 128.0f;", False),
    ("int8 rounding toward zero", "float q = rintf((float)x[i] / s);", "float q = truncf((float)x[i] / s);", False),
    ("int8 quotient in fp64", "float q = rintf((float)x[i] / s);", "float q = (float)rint(x[i] / (double)s);", False),
    ("e4m3 four mantissa bits", "int q = (e - 1) - 3;", "int q = (e - 1) - 4;", False),
    ("e4m3 no saturation", "if (r > 448.0) r = 448.0;", "if (r > 480.0) r = 480.0;", False),
    ("e4m3 ties away from zero", "double r = rint(a / ldexp(1.0, q)) * ldexp(1.0, q);",
     "double r = floor(a / ldexp(1.0, q) + 0.5) * ldexp(1.0, q);", False),
    ("e4m3 subnormal spacing", "if (q < -9) q = -9;", "if (q < -10) q = -10;", False),
    ("e4m3 group scale over 480", "float s = amax / 448.0f;", "float s = amax / 480.0f;", False),
    ("e4m3 quotient in fp64", "round_e4m3((double)((float)xg[i] / s))", "round_e4m3(xg[i] / (double)s)", False),
    ("append rotates values", "const double *vs = v_new + (t * heads + h) * (int64_t)d;",
     "const double *vs = krow - (int64_t)0 * (t * heads + h);", False),
]


@pytest.mark.parametrize("name,old,new,every", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new, every):
    text = open(SRC).read()
    assert old in text, f"mutation site for '{name}' not found"
    text = text.replace(old, new) if every else text.replace(old, new, 1)
    src = tmp_path / "oracle_mutant.c"
    src.write_text(text)
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", str(src),
                           "-o", str(lib), "-lm"])
    env = dict(os.environ, ORACLE_LIB=str(lib), OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant '{name}' survived the pin suite:\n{r.stdout[-2000:]}"
