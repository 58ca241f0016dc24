"""The oracle pins must reject plausible mistakes.

Each case plants one mistake (a dropped term, a wrong factor, a wrong index,
a wrong sign) in a temporary copy of the oracle's C source, builds it, and
runs the pin suite against that copy: at least one pin has to fail.  The
committed oracle itself is never modified.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "polar_oracle.c")

MUTANTS = {
    "temperature_without_floor": ("return t > 1.0 ? t : 1.0;", "return t;"),
    "temperature_from_T_not_n": ("double tau = temperature(n, jb->c);",
                                 "double tau = temperature(jb->T, jb->c);"),
    "neff_drops_square": ("double ne = st->l * st->l / st->q2;",
                          "double ne = st->l / st->q2;"),
    "stream_unsquared_correction": ("st->q2 *= alpha * alpha;",
                                    "st->q2 *= alpha;"),
    "merge_unsquared_weight": ("dst->q2 += w * w * parts[s].q2;",
                               "dst->q2 += w * parts[s].q2;"),
    "floor_missing_two": ("double r = sqrt(2.0 * log((double)n));",
                          "double r = sqrt(log((double)n));"),
    "second_order_floor_without_gamma": (
        "(2.0 * r) + EULER_GAMMA / r);", "(2.0 * r));"),
    "floor_missing_temperature": (
        "double sigma = tau * c->sigma_k * qn / sqrt((double)d);",
        "double sigma = c->sigma_k * qn / sqrt((double)d);"),
    "lse_wrong_sign": ("double lse = st->m + log(st->l);",
                       "double lse = st->m - log(st->l);"),
    "count_ungated": ("*count = cf * tanh(log(ne) / c->kappa);",
                      "*count = tanh(log(ne) / c->kappa);"),
    "memory_dropped": ("o[x] = u[x] + cnt * jb->w[x] + mi[x];",
                       "o[x] = u[x] + cnt * jb->w[x];"),
    "key_row_index": ("s[j] = scale * dot(q, K + j * d, d);",
                      "s[j] = scale * dot(q, K + j, d);"),
    # the unit-sphere guard taken on |acc| = l |a| instead of |a|
    "direction_guard_on_unnormalised_acc": (
        "double den = an > c->eps ? an : c->eps;",
        "double den = an * st->l > c->eps ? an : c->eps / st->l;"),
    "direction_guard_additive": ("double den = an > c->eps ? an : c->eps;",
                                 "double den = an + c->eps;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o",
                           str(lib), str(mut), "-lm", "-lpthread"])
    env = dict(os.environ, POLAR_ORACLE_LIB=str(lib))
    r = subprocess.run(
        [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
         os.path.join(ROOT, "tests", "test_oracle_pins.py")],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins accepted mutant {name}:\n{r.stdout[-2000:]}"
