"""The pins must catch plausible mistakes in the oracle.

Each case plants one mistake in a copy of oracle/ldn_oracle.c (a sign, a
dropped factor, a transposed index, a wrong operand), builds it into a
temporary library on the CPU, and runs the pin suite against it in a child
process.  The pin suite must fail for every mutant.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ldn_oracle.c")

MUTANTS = {
    # the error is written with the wrong sign
    "update_sign": ("W[(size_t)i * dk + c] += r * (double)k[c];",
                    "W[(size_t)i * dk + c] -= r * (double)k[c];"),
    # the write strength beta is dropped
    "drop_beta": ("const double r = beta * (", "const double r = 1.0 * ("),
    # the scalar forget gate is ignored
    "drop_alpha": ("const double alpha = exp((double)J->gate[tok]);", "const double alpha = 1.0;"),
    # the per-channel decay acts on the value side instead of the key side
    "kda_left": ("const double a = exp((double)g[c]);\n                for (int i = 0; i < dv; ++i) W[(size_t)i * dk + c] *= a;",
                 "for (int i = 0; i < dv; ++i) W[(size_t)i * dk + c] *= exp((double)g[i % dk]);"),
    # the output reads the memory with the key instead of the query
    "read_with_key": ("s += W[(size_t)i * dk + c] * (double)q[c];",
                      "s += W[(size_t)i * dk + c] * (double)k[c];"),
    # the initial state is read without the transpose
    "s0_orientation": ("W[(size_t)i * dk + c] = (double)s0[(size_t)c * dv + i];",
                       "W[(size_t)i * dk + c] = (double)s0[(size_t)i * dk + c];"),
    # the prediction uses the query instead of the key
    "predict_with_query": ("s += W[(size_t)i * dk + c] * (gdn2 ? (double)eb[c] * (double)k[c] : (double)k[c]);",
                           "s += W[(size_t)i * dk + c] * (gdn2 ? (double)eb[c] * (double)k[c] : (double)q[c]);"),
    # Gated DeltaNet-2: the erase gate is not applied to the prediction direction
    "gdn2_no_erase": ("(gdn2 ? (double)eb[c] * (double)k[c] : (double)k[c])", "(double)k[c]"),
    # Gated DeltaNet-2: the write gate is not applied to the value
    "gdn2_no_write": ("const double target = gdn2 ? (double)ww[i] * (double)v[i] : (double)v[i];",
                      "const double target = (double)v[i];"),
    # GDN2: the write goes along the erase direction e = b * k instead of k (the notes
    # single this out: the outer product keeps k)
    "gdn2_write_along_erase": ("for (int c = 0; c < dk; ++c) W[(size_t)i * dk + c] += r * (double)k[c];",
                               "for (int c = 0; c < dk; ++c) W[(size_t)i * dk + c] += r * (gdn2 ? (double)eb[c] * "
                               "(double)k[c] : (double)k[c]);"),
    # RLA / RDN: the residual read from the decayed base state instead of the old one
    "rla_residual_decayed": ("double r = (double)v[i] - pk;", "double r = (double)v[i] - alpha * pk;"),
    # RLA / RDN: the correction read without its gamma
    "rla_output_no_gamma": ("o[i] += gamma * rq;", "o[i] += rq;"),
    # RLA / RDN: the residual clipped from above only
    "rla_clip_one_sided": ("if (r < -clip) r = -clip;", "(void)0;"),
    # RDN: the residual state's delta correction without the decay
    "rdn_correction_undecayed": ("const double w = gamma * (tmp[i] - (J->delta ? alpha * rk : 0.0));",
                                 "const double w = gamma * (tmp[i] - (J->delta ? rk : 0.0));"),
    # backward: the key gradient misses its write term (G^T r)
    "bwd_dk_no_write": ("s += G[(size_t)i * dk + c] * r[i] + Wt[(size_t)i * dk + c] * dp[i];",
                        "s += Wt[(size_t)i * dk + c] * dp[i];"),
    # backward: the prediction's gradient with the wrong sign
    "bwd_dp_sign": ("dp[i] = -beta * dr;", "dp[i] = beta * dr;"),
    # backward: the query gradient read from the state before the write
    "bwd_dq_pre_write": ("for (int i = 0; i < dv; ++i) s += W[(size_t)i * dk + c] * (double)dO[i];",
                         "for (int i = 0; i < dv; ++i) s += Wt[(size_t)i * dk + c] * (double)dO[i];"),
    # backward: the state gradient not carried through the scalar decay
    "bwd_no_decay": ("for (size_t x = 0; x < D2; ++x) G[x] *= a_t;", "(void)a_t;"),
    # backward: the per-channel decay gradient taken against the state before the decay
    "bwd_dg_wrong_state": ("for (int i = 0; i < dv; ++i) s += G[(size_t)i * dk + c] * Wt[(size_t)i * dk + c];",
                           "for (int i = 0; i < dv; ++i) s += G[(size_t)i * dk + c] * Wt[(size_t)i * dk + c] * exp(-(double)g[c]) * 0.5;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutant_c = tmp_path / "mutant.c"
    mutant_c.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    "-D_POSIX_C_SOURCE=200809L", str(mutant_c), "-o", str(lib), "-lm"], check=True)
    env = dict(os.environ, LDN_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        os.path.join(ROOT, "tests", "test_gdn2_oracle_pins.py"),
                        os.path.join(ROOT, "tests", "test_bwd_oracle_pins.py"),
                        os.path.join(ROOT, "tests", "test_rla_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
