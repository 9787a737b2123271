"""The pins must catch plausible mistakes in the oracle.

Each mutant is a copy of the oracle source with one deliberate slip, built on
the CPU into a temporary library; the pin and brute-force suites are then run
against it in a subprocess and must fail."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "adafactor_oracle.c")

MUTANTS = {
    "row mean drops eps1": ("for (int64_t j = 0; j < W; ++j) s += gb[i * W + j] * gb[i * W + j] + hp->eps1;",
                            "for (int64_t j = 0; j < W; ++j) s += gb[i * W + j] * gb[i * W + j];"),
    "EMA coefficients swapped": ("rb[i] = beta2 * rb[i] + (1.0 - beta2) * (s / (double)W);",
                                 "rb[i] = (1.0 - beta2) * rb[i] + beta2 * (s / (double)W);"),
    "beta2 exponent sign": ("return 1.0 - pow((double)t, hp->decay_rate);",
                            "return 1.0 - pow((double)t, -hp->decay_rate);"),
    "no mean(row) normalisation": ("double r_fac = 1.0 / sqrt(rb[i] / m);", "double r_fac = 1.0 / sqrt(rb[i]);"),
    "column mean over the wrong axis": ("(colsum[j] / (double)H)", "(colsum[j] / (double)W)"),
    "clip divides instead of multiplies": ("double clip_div = rms(u, n) / hp->clip_threshold;",
                                           "double clip_div = rms(u, n) * hp->clip_threshold;"),
    "clip never active": ("if (clip_div < 1.0) clip_div = 1.0;", "clip_div = 1.0;"),
    "no eps2 floor on RMS(p)": ("alpha = rho * (hp->eps2 > r ? hp->eps2 : r);", "alpha = rho * r;"),
    "relative step cap 1e-3": ("double cap = hp->warmup_init ? 1e-6 * (double)t : 1e-2;",
                               "double cap = hp->warmup_init ? 1e-6 * (double)t : 1e-3;"),
    "warmup cap not scaled by t": ("double cap = hp->warmup_init ? 1e-6 * (double)t : 1e-2;",
                                   "double cap = hp->warmup_init ? 1e-6 : 1e-2;"),
    "beta1 coefficients swapped": ("exp_avg[k] = hp->beta1 * exp_avg[k] + (1.0 - hp->beta1) * u[k];",
                                   "exp_avg[k] = (1.0 - hp->beta1) * exp_avg[k] + hp->beta1 * u[k];"),
    "weight decay not scaled by the lr": ("p[k] = p[k] - hp->weight_decay * alpha * p[k];",
                                          "p[k] = p[k] - hp->weight_decay * p[k];"),
    "unfactored update without sqrt": ("u[k] = g[k] / sqrt(v[k]);", "u[k] = g[k] / v[k];"),
    "RMS without the mean": ("return sqrt(s / (double)n);", "return sqrt(s);"),
    "update not scaled by lr": ("u[k] = (u[k] / clip_div) * alpha;", "u[k] = (u[k] / clip_div);"),
    "exp_avg not used as the update": ("u[k] = exp_avg[k];", "(void)0;"),
    "8-bit codes floored": ("q = rintf(x);", "q = floorf(x);"),
    "8-bit ties rounded away from zero": ("q = rintf(x);", "q = roundf(x);"),
    "8-bit code by the reciprocal of the scale": (
        "const float x = (float)moment[r * last + j] / scale;",
        "const float x = (float)moment[r * last + j] * (127.0f / amax);"),
    "8-bit scale over 128": ("const float scale = amax / 127.0f;", "const float scale = amax / 128.0f;"),
    "8-bit groups flat across rows": ("*last = ndim >= 2 ? shape[ndim - 1] : n;", "*last = n;"),
    "8-bit update from the unquantised moment": ("oracle_q8_apply(p, ndim, shape, codes, scales, alpha, hp);",
                                                 "apply_update(p, m, n, alpha, hp);"),
    "8-bit old moment without its scale": ("const float x = (float)code * scale;", "const float x = (float)code;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found once: {old}"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", str(mut),
                           "-o", str(lib), "-lm"])
    env = dict(os.environ, ORACLE_LIB_OVERRIDE=str(lib))
    res = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                          os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                          os.path.join(ROOT, "tests", "test_oracle_q8_pins.py"),
                          os.path.join(ROOT, "tests", "test_oracle_bruteforce.py")],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode != 0, f"mutant '{name}' survived the pins:\n{res.stdout[-2000:]}"


LAMB_SRC = os.path.join(ROOT, "oracle", "lamb_oracle.c")
LAMB_MUTANTS = {
    "bias correction with power t + 1": ("1.0 - pow(hp->beta1, (double)t)", "1.0 - pow(hp->beta1, (double)(t + 1))"),
    "second-moment EMA coefficients swapped": (
        "v[i] = hp->beta2 * v[i] + (1.0 - hp->beta2) * g[i] * g[i];",
        "v[i] = (1.0 - hp->beta2) * v[i] + hp->beta2 * g[i] * g[i];"),
    "no square root of vh": ("return mh / (sqrt(vh) + hp->eps) + hp->weight_decay * p;",
                             "return mh / (vh + hp->eps) + hp->weight_decay * p;"),
    "eps inside the square root": ("return mh / (sqrt(vh) + hp->eps) + hp->weight_decay * p;",
                                   "return mh / sqrt(vh + hp->eps) + hp->weight_decay * p;"),
    "trust ratio inverted": ("? pn / rn : 1.0;", "? rn / pn : 1.0;"),
    "zero norm gives trust 0": ("? pn / rn : 1.0;", "? pn / rn : 0.0;"),
    "weight decay left out of the direction": ("return mh / (sqrt(vh) + hp->eps) + hp->weight_decay * p;",
                                               "return mh / (sqrt(vh) + hp->eps);"),
    "lr not applied": ("p[i] = p[i] - hp->lr * trust * r;", "p[i] = p[i] - trust * r;"),
}


@pytest.mark.parametrize("name", sorted(LAMB_MUTANTS))
def test_lamb_pins_catch_mutant(name, tmp_path):
    old, new = LAMB_MUTANTS[name]
    src = open(LAMB_SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found once: {old}"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", str(mut),
                           "-o", str(lib), "-lm"])
    env = dict(os.environ, ORACLE_LAMB_LIB_OVERRIDE=str(lib))
    res = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                          os.path.join(ROOT, "tests", "test_oracle_lamb_pins.py")],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode != 0, f"mutant '{name}' survived the pins:\n{res.stdout[-2000:]}"


CAME_SRC = os.path.join(ROOT, "oracle", "came_oracle.c")
CAME_MUTANTS = {
    "instability against the old momentum": (
        """        exp_avg[k] = hp->beta1 * exp_avg[k] + (1.0 - hp->beta1) * u[k];
        const double dlt = u[k] - exp_avg[k];""",
        """        const double dlt = u[k] - exp_avg[k];
        exp_avg[k] = hp->beta1 * exp_avg[k] + (1.0 - hp->beta1) * u[k];"""),
    "eps2 dropped": ("x[k] = dlt * dlt + hp->eps2;", "x[k] = dlt * dlt;"),
    "beta2 used for the instability": ("hp->beta3, res_row + b * H", "hp->beta2, res_row + b * H"),
    "no mean normalisation of the factors": ("f[i * W + j] = rb[i] * cb[j] / mr;", "f[i * W + j] = rb[i] * cb[j];"),
    "column mean over the wrong axis": ("cb[j] = beta * cb[j] + (1.0 - beta) * (s / (double)H);",
                                        "cb[j] = beta * cb[j] + (1.0 - beta) * (s / (double)W);"),
    "clip inverted": ("double clip_div = rms(u, n) / hp->clip_threshold;",
                      "double clip_div = rms(u, n) * hp->clip_threshold;"),
    "no square root of S": ("p[k] = p[k] - hp->lr * exp_avg[k] / sqrt(f[k]);",
                            "p[k] = p[k] - hp->lr * exp_avg[k] / f[k];"),
    "weight decay without the lr": ("p[k] = p[k] - hp->weight_decay * hp->lr * p[k];",
                                    "p[k] = p[k] - hp->weight_decay * p[k];"),
    "momentum coefficients swapped": ("exp_avg[k] = hp->beta1 * exp_avg[k] + (1.0 - hp->beta1) * u[k];",
                                      "exp_avg[k] = (1.0 - hp->beta1) * exp_avg[k] + hp->beta1 * u[k];"),
    "vector path without eps1": ("for (int64_t k = 0; k < n; ++k) x[k] = g[k] * g[k] + hp->eps1;",
                                 "for (int64_t k = 0; k < n; ++k) x[k] = g[k] * g[k];"),
}


@pytest.mark.parametrize("name", sorted(CAME_MUTANTS))
def test_came_pins_catch_mutant(name, tmp_path):
    old, new = CAME_MUTANTS[name]
    src = open(CAME_SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found once: {old}"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", str(mut),
                           "-o", str(lib), "-lm"])
    env = dict(os.environ, ORACLE_CAME_LIB_OVERRIDE=str(lib))
    res = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                          os.path.join(ROOT, "tests", "test_oracle_came_pins.py"),
                          os.path.join(ROOT, "tests", "test_oracle_came_bruteforce.py")],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode != 0, f"mutant '{name}' survived the pins:\n{res.stdout[-2000:]}"
