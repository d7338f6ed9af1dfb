"""The oracle's native self-test (oracle/ldn_oracle_selftest.c): the worked
example of the linear-attention notes (Sec. 2.3), the exact write at beta = 1,
a brute force by explicit 4 x 4 matrices, the mode reductions and state passing,
checked in C without numpy.  It must pass on the oracle as built, and fail on
plausible mistakes planted in a copy of the oracle's forward recurrence."""
import os
import subprocess

import pytest

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "ldn_oracle.c")

# mistakes in the forward recurrence (one line each); the Python pin suite is run
# against the same mutants in test_oracle_mutations.py
FORWARD_MUTANTS = {
    "update_sign": ("W[(size_t)i * dk + c] += r * (double)k[c];", "W[(size_t)i * dk + c] -= r * (double)k[c];"),
    "drop_beta": ("const double r = beta * (", "const double r = 1.0 * ("),
    "drop_alpha": ("const double alpha = exp((double)J->gate[tok]);", "const double alpha = 1.0;"),
    "read_with_key": ("s += W[(size_t)i * dk + c] * (double)q[c];", "s += W[(size_t)i * dk + c] * (double)k[c];"),
    "s0_orientation": ("W[(size_t)i * dk + c] = (double)s0[(size_t)c * dv + i];",
                       "W[(size_t)i * dk + c] = (double)s0[(size_t)i * dk + c];"),
    "predict_with_query": ("s += W[(size_t)i * dk + c] * (gdn2 ? (double)eb[c] * (double)k[c] : (double)k[c]);",
                           "s += W[(size_t)i * dk + c] * (gdn2 ? (double)eb[c] * (double)k[c] : (double)q[c]);"),
    "kda_left": ("const double a = exp((double)g[c]);\n                for (int i = 0; i < dv; ++i) W[(size_t)i * dk + c] *= a;",
                 "for (int i = 0; i < dv; ++i) W[(size_t)i * dk + c] *= exp((double)g[i % dk]);"),
}


def test_selftest_passes():
    exe = oracle.build_selftest()
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "0 failure(s)" in r.stdout and "FAIL" not in r.stdout


@pytest.mark.parametrize("name", sorted(FORWARD_MUTANTS))
def test_selftest_catches_mutant(name, tmp_path):
    old, new = FORWARD_MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new))
    exe = oracle.build_selftest(oracle_src=str(mutant), out=str(tmp_path / "selftest"))
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode != 0, f"mutant {name} passed the native self-test:\n{r.stdout}"
