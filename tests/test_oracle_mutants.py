"""The oracle's pins catch plausible mistakes.  Each case plants one mistake
in a copy of the oracle's C source (a dropped, added or misplaced eps, a
transposed index, a wrong mean, a swapped scale group, ties rounded away from
zero, a flattening in the wrong order, ...), builds the copy in a temporary
directory and runs the pin tests against it: at least one pin must fail.
The control case runs the same harness on an unmodified copy, which must
pass, so a failure is the planted mistake's and not the harness's.

CPU only; the mistakes are planted in the oracle, never in the product."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.join(ROOT, "tests")
MAIN_PINS = [os.path.join(TESTS, "test_oracle_pins.py"),
             os.path.join(TESTS, "test_oracle_head_pins.py")]
MX_PINS = [os.path.join(TESTS, "test_oracle_mxfp8_pins.py")]

STATS_RSQ = "double r = 1.0 / sqrt(ss / (double)O_K + rms_eps);"

# (name, text in mhc_oracle.c, replacement, pin files)
MUTANTS = [
    ("stats: eps outside the sqrt", STATS_RSQ,
     "double r = 1.0 / (sqrt(ss / (double)O_K) + rms_eps);", MAIN_PINS),
    ("stats: mean over one stream", STATS_RSQ,
     "double r = 1.0 / sqrt(ss / (double)O_H + rms_eps);", MAIN_PINS),
    ("stats: row flattened hidden-major",
     "x[k] = oracle_bf16_to_double(row[k]);\n            ss += x[k] * x[k];\n        }\n        "
     + STATS_RSQ,
     "x[k] = oracle_bf16_to_double(row[(k % O_HC) * O_H + k / O_HC]);\n            "
     "ss += x[k] * x[k];\n        }\n        " + STATS_RSQ, MAIN_PINS),
    ("split: post and comb scales swapped", "int g = c < 4 ? 0 : (c < 8 ? 1 : 2);",
     "int g = c < 4 ? 0 : (c < 8 ? 2 : 1);", MAIN_PINS),
    ("split: pre without eps", "pre[m * O_HC + i] = sigmoid(l[i]) + pre_eps;",
     "pre[m * O_HC + i] = sigmoid(l[i]);", MAIN_PINS),
    ("split: post with eps", "post[m * O_HC + i] = post_mult * sigmoid(l[4 + i]);",
     "post[m * O_HC + i] = post_mult * sigmoid(l[4 + i]) + pre_eps;", MAIN_PINS),
    ("split: comb block transposed", "C[j][i] = exp(l[8 + 4 * j + i]);",
     "C[j][i] = exp(l[8 + 4 * i + j]);", MAIN_PINS),
    ("sinkhorn: column step without eps",
     "for (int j = 0; j < O_HC; ++j)\n                    C[j][i] = C[j][i] / (s + sink_eps);",
     "for (int j = 0; j < O_HC; ++j)\n                    C[j][i] = C[j][i] / s;", MAIN_PINS),
    ("sinkhorn: row step with twice the eps",
     "for (int i = 0; i < O_HC; ++i)\n                    C[j][i] = C[j][i] / (s + sink_eps);",
     "for (int i = 0; i < O_HC; ++i)\n                    C[j][i] = C[j][i] / (s + 2 * sink_eps);",
     MAIN_PINS),
    ("combine: norm mean over 4 streams",
     "double rn = 1.0 / sqrt(ss / (double)O_H + norm_eps);",
     "double rn = 1.0 / sqrt(ss / (double)O_K + norm_eps);", MAIN_PINS),
    ("combine: norm weight dropped",
     "oracle_double_to_bf16(y[h] * rn * oracle_bf16_to_double(w[h]));",
     "oracle_double_to_bf16(y[h] * rn);", MAIN_PINS),
    ("combine: streams interleaved",
     "acc += pre[m * O_HC + i] * oracle_bf16_to_double(row[i * O_H + h]);",
     "acc += pre[m * O_HC + i] * oracle_bf16_to_double(row[h * O_HC + i]);", MAIN_PINS),
    ("combine: every row gated by row 0",
     "acc += pre[m * O_HC + i] * oracle_bf16_to_double(row[i * O_H + h]);",
     "acc += pre[i] * oracle_bf16_to_double(row[i * O_H + h]);", MAIN_PINS),
    ("sinkhorn: one iteration short", "for (int t = 0; t < iters; ++t)",
     "for (int t = 0; t < iters - 1; ++t)", MAIN_PINS),
    ("split: logit without base",
     "l[c] = mix[m * O_MIX + c] * (double)scale[g] + (double)base[c];",
     "l[c] = mix[m * O_MIX + c] * (double)scale[g];", MAIN_PINS),
    ("stats: mix divided by rsqrt", "mix[m * O_MIX + c] = dot * r;",
     "mix[m * O_MIX + c] = dot / r;", MAIN_PINS),
    ("bf16: subnormals flushed", "    if (q < -133)\n        q = -133;",
     "    if (q < -126)\n        q = -126;", MAIN_PINS),
    ("hc_head: streams interleaved", "acc += p[i] * x[i * O_H + h];",
     "acc += p[i] * x[h * O_HC + i];", MAIN_PINS),
    ("post: every row gated by row 0", "double p = (double)post[m * O_HC + i];",
     "double p = (double)post[i];", MAIN_PINS),
    ("post: comb transposed", "acc += (double)comb[m * 16 + j * 4 + i] *",
     "acc += (double)comb[m * 16 + i * 4 + j] *", MAIN_PINS),
    ("post: sublayer output dropped", "double acc = p * oracle_bf16_to_double(yr[h]);",
     "double acc = 0.0 * p;", MAIN_PINS),
    ("bf16: ties away from zero", "double r = nearbyint(s);", "double r = round(s);", MAIN_PINS),
    ("hc_head: eps inside the sigmoid",
     "p[c] = sigmoid(mx * (double)scale[0] + (double)base[c]) + hc_eps;",
     "p[c] = sigmoid(mx * (double)scale[0] + (double)base[c] + hc_eps);", MAIN_PINS),
    ("hc_head: rsqrt without eps", "double r = 1.0 / sqrt(ss / (double)O_K + norm_eps);",
     "double r = 1.0 / sqrt(ss / (double)O_K);", MAIN_PINS),
    ("stats: every row's mix in row 0", "mix[m * O_MIX + c] = dot * r;", "mix[c] = dot * r;",
     MAIN_PINS),
    ("split: every row's pre in row 0", "pre[m * O_HC + i] = sigmoid(l[i]) + pre_eps;",
     "pre[i] = sigmoid(l[i]) + pre_eps;", MAIN_PINS),
    ("stats: fn row stride dropped",
     "const float *f = fn + (int64_t)c * O_K;\n            double dot = 0.0;\n            "
     "for (int k = 0; k < O_K; ++k)\n                dot += x[k] * (double)f[k];\n            "
     "mix[m * O_MIX + c]",
     "const float *f = fn + (int64_t)c;\n            double dot = 0.0;\n            "
     "for (int k = 0; k < O_K; ++k)\n                dot += x[k] * (double)f[k];\n            "
     "mix[m * O_MIX + c]", MAIN_PINS),
    ("sinkhorn: row step sums a column",
     "for (int i = 0; i < O_HC; ++i)\n                    s += C[j][i];",
     "for (int i = 0; i < O_HC; ++i)\n                    s += C[i][j];", MAIN_PINS),
    ("post: output streams interleaved",
     "R_out[m * (int64_t)O_K + i * O_H + h] = oracle_double_to_bf16(acc);",
     "R_out[m * (int64_t)O_K + i + h * O_HC] = oracle_double_to_bf16(acc);", MAIN_PINS),
    ("split: comb written transposed", "comb[m * 16 + j * 4 + i] = C[j][i];",
     "comb[m * 16 + j * 4 + i] = C[i][j];", MAIN_PINS),
    ("combine: eps outside the sqrt", "double rn = 1.0 / sqrt(ss / (double)O_H + norm_eps);",
     "double rn = 1.0 / (sqrt(ss / (double)O_H) + norm_eps);", MAIN_PINS),
    ("mxfp8: scale exponent off by one", "e = (ex - 1) - 8;", "e = ex - 8;", MX_PINS),
    ("mxfp8: ties away from zero", "double t = ldexp(nearbyint(ldexp(a, -q)), q);",
     "double t = ldexp(round(ldexp(a, -q)), q);", MX_PINS),
    ("mxfp8: no saturation", "    if (t > 448.0)\n        t = 448.0;\n", "", MX_PINS),
    ("mxfp8: sign of -0 lost", "uint8_t sign = signbit(v) ? 0x80 : 0;",
     "uint8_t sign = v < 0 ? 0x80 : 0;", MX_PINS),
    ("mxfp8: subnormal quantum", "q = -9;                   /* subnormal quantum */", "q = -10;",
     MX_PINS),
    ("mxfp8: tile rows swapped",
     "int64_t inner = (m % 32) * 16 + ((m % 128) / 32) * 4 + g % 4;",
     "int64_t inner = ((m % 128) / 32) * 128 + (m % 32) * 4 + g % 4;", MX_PINS),
]


def _run_pins(tmp_path, source, pins):
    copy = tmp_path / "oracle"
    shutil.copytree(os.path.join(ROOT, "oracle"), copy,
                    ignore=shutil.ignore_patterns("_build", "__pycache__"))
    (copy / "mhc_oracle.c").write_text(source)
    # the copy comes first on the path; the tests' conftest then leaves it there
    env = dict(os.environ, PYTHONPATH=str(tmp_path) + os.pathsep + ROOT)
    return subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                           *pins], cwd=str(tmp_path), env=env, capture_output=True, text=True,
                          timeout=900)


def _source():
    with open(os.path.join(ROOT, "oracle", "mhc_oracle.c")) as f:
        return f.read()


def test_unmodified_copy_passes_the_pins(tmp_path):
    out = _run_pins(tmp_path, _source(), MAIN_PINS + MX_PINS)
    assert out.returncode == 0, out.stdout[-3000:]


@pytest.mark.parametrize("name,old,new,pins", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(tmp_path, name, old, new, pins):
    src = _source()
    assert src.count(old) == 1, f"{name}: the text to mutate is not unique"
    out = _run_pins(tmp_path, src.replace(old, new), pins)
    # 1: tests ran and at least one failed (not an import or collection error)
    assert out.returncode == 1, f"{name}: no pin failed\n" + out.stdout[-3000:]
