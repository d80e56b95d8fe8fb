"""The oracle pins must reject a broken oracle.

Each case plants one plausible mistake in a scratch copy of oracle.c (never in
the committed file), builds it, and runs the pin suite against that build in a
subprocess.  Every mutant must fail at least one pin.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "drop_skip_term": ("yt[d] = acc + j->D[h] * xt[d];", "yt[d] = acc;"),
    "swap_B_and_C": ("Sd[n] = decay * Sd[n] + v * Bt[n];\n        acc += Sd[n] * Ct[n];",
                     "Sd[n] = decay * Sd[n] + v * Ct[n];\n        acc += Sd[n] * Bt[n];"),
    "group_index_mod": ("const int g = h / (H / G);", "const int g = h % G;"),
    "decay_sign": ("exp(delta * j->A[h])", "exp(-delta * j->A[h])"),
    "exp_instead_of_softplus": ("const double delta = softplus64(j->dt[t * H + h] + j->dt_bias[h]);",
                                "const double delta = exp(j->dt[t * H + h] + j->dt_bias[h]);"),
    "output_before_update": ("        Sd[n] = decay * Sd[n] + v * Bt[n];\n        acc += Sd[n] * Ct[n];",
                             "        acc += Sd[n] * Ct[n];\n        Sd[n] = decay * Sd[n] + v * Bt[n];"),
    "missing_dt_bias": ("softplus64(j->dt[t * H + h] + j->dt_bias[h])", "softplus64(j->dt[t * H + h])"),
    "initial_state_ignored": ("  double* S = j->state + ((int64_t)s * H + h) * (int64_t)P * N;\n",
                              "  double* S = j->state + ((int64_t)s * H + h) * (int64_t)P * N;\n"
                              "  memset(S, 0, sizeof(double) * (size_t)P * N);\n"),
    "state_of_sequence_zero": ("double* S = j->state + ((int64_t)s * H + h) * (int64_t)P * N;",
                               "double* S = j->state + ((int64_t)0 * H + h) * (int64_t)P * N;"),
    "first_token_skipped": ("for (int64_t t = j->cu[s]; t < j->cu[s + 1]; ++t) {",
                            "for (int64_t t = j->cu[s] + 1; t < j->cu[s + 1]; ++t) {"),
    "skip_term_head_zero": ("yt[d] = acc + j->D[h] * xt[d];", "yt[d] = acc + j->D[0] * xt[d];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(SRC).read()
    assert before in src, "mutation site no longer present in oracle.c"
    mut_c = tmp_path / "oracle_mut.c"
    mut_c.write_text(src.replace(before, after))
    so = tmp_path / "oracle_mut.so"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-o", str(so), str(mut_c), "-lm", "-lpthread"])
    env = dict(os.environ, ERS_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
