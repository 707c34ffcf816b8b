"""Mutation check of the oracle's pins (CPU).

Each case plants one plausible mistake in a copy of oracle/rlcs_oracle.c:
a dropped factor, a wrong index, a swapped clip, a misplaced reset. The copy
is compiled to a temporary library, and the oracle pin suite
(test_oracle_pins.py) runs against it. Every mutant must make at least one
pin fail: a mutant that survives means the pins have a blind spot. The
mistakes are planted in the oracle on the CPU only.
"""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "rlcs_oracle.c")

MUTANTS = {
    "gae_drops_lambda": ("a += gamma * lambda * a_next;", "a += gamma * a_next;"),
    "gae_delta_sign": ("double delta = (double)r[t] + gamma * s - (double)v[t];",
                       "double delta = (double)r[t] + gamma * s + (double)v[t];"),
    "successor_same_step": ("return (double)values[t + 1];", "return (double)values[t];"),
    "terminated_takes_bootstrap": ("if (SET(term, t)) return 0.0;", "if (SET(term, t)) return boot;"),
    "truncation_wins": (
        "  if (SET(term, t)) return 0.0;\n  if (trunc != NULL && SET(trunc, t)) return (double)next_values[t];",
        "  if (trunc != NULL && SET(trunc, t)) return (double)next_values[t];\n  if (SET(term, t)) return 0.0;"),
    "bootstrap_dropped": ("if (t == T - 1) return boot;", "if (t == T - 1) return 0.0;"),
    "lambda_return_weights_swapped": ("gamma * ((1.0 - lambda) * (double)v[t + 1] + lambda * g_next);",
                                      "gamma * (lambda * (double)v[t + 1] + (1.0 - lambda) * g_next);"),
    "discount_missing": ("g = (double)r[t] + gamma * g_next;", "g = (double)r[t] + g_next;"),
    "vtrace_c_uses_rho_bar": ("double c = lambda * fmin(c_bar, ratio);",
                              "double c = lambda * fmin(rho_bar, ratio);"),
    "vtrace_drops_lambda": ("double c = lambda * fmin(c_bar, ratio);", "double c = fmin(c_bar, ratio);"),
    "vtrace_pg_uses_own_vs": ("double w = cut ? s : vs_next;", "double w = cut ? s : vs_t;"),
    "retrace_trace_same_step": ("double c_next = lambda * fmin(c_bar, exp((double)lr[t + 1]));",
                                "double c_next = lambda * fmin(c_bar, exp((double)lr[t]));"),
    "retrace_drops_q": ("c_next * (qret_next - (double)q[t + 1]));", "c_next * qret_next);"),
    "elig_reset_same_step": ("if (t > 0 && !SET(d, t - 1)) e += gamma * lambda * e_prev;",
                             "if (!SET(d, t)) e += gamma * lambda * e_prev;"),
    "psum_no_reset": ("if (t > 0 && !SET(d, t - 1)) s += s_prev;", "if (t > 0) s += s_prev;"),
    "affine_reset_ignored": ("if (rr == NULL || !SET(rr, t)) v += (double)ar[t] * prev;",
                             "v += (double)ar[t] * prev;"),
    "affine_init_dropped": ("double prev = x_init ? (double)x_init[n] : 0.0;", "double prev = 0.0;"),
    "psum_reset_same_step": ("if (t > 0 && !SET(d, t - 1)) s += s_prev;",
                             "if (t > 0 && !SET(d, t)) s += s_prev;"),
    "truncation_does_not_cut": ("  if (trunc != NULL && SET(trunc, t)) return 1;",
                                "  if (trunc != NULL && SET(trunc, t)) return 0;"),
    "gae_carries_across_cut": ("if (!is_cut(d, tr, t, T)) a += gamma * lambda * a_next;",
                               "a += gamma * lambda * a_next;"),
    "vtrace_rho_uses_c_bar": ("double rho = fmin(rho_bar, ratio);", "double rho = fmin(c_bar, ratio);"),
    "vtrace_pg_drops_rho": ("pg_row[t] = rho * ((double)r[t] + gamma * w - (double)v[t]);",
                            "pg_row[t] = (double)r[t] + gamma * w - (double)v[t];"),
    "vtrace_diff_uses_own_value": ("if (!cut) diff += gamma * c * (vs_next - v_next);",
                                   "if (!cut) diff += gamma * c * (vs_next - (double)v[t]);"),
    "elig_drops_gamma": ("if (t > 0 && !SET(d, t - 1)) e += gamma * lambda * e_prev;",
                         "if (t > 0 && !SET(d, t - 1)) e += lambda * e_prev;"),
    "affine_direction_ignored": ("int64_t t = reverse ? T - 1 - i : i;", "int64_t t = i;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation site not found exactly once: %s" % name
    mutated = src.replace(old, new)
    c_path = tmp_path / "mutant.c"
    so_path = tmp_path / "libmutant.so"
    c_path.write_text(mutated)
    subprocess.run(["gcc", "-std=c99", "-O1", "-ffp-contract=off", "-fPIC", "-shared",
                    str(c_path), "-o", str(so_path), "-lm"], check=True)
    env = dict(os.environ, RLCS_ORACLE_LIB=str(so_path))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "mutant %s survived the oracle pins:\n%s" % (name, r.stdout[-2000:])
