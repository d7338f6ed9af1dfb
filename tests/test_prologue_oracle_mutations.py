"""The prologue / epilogue pins must catch plausible mistakes in that oracle.

Each case plants one mistake in a copy of oracle/prologue.py (a reversed or
shifted convolution kernel, eps outside the root, a sign, a dropped factor, a
sum for a mean), places it as the `oracle` package of a temporary directory,
and runs tests/test_prologue_oracle_pins.py against it in a child process.  The
pins must fail for every mutant."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "prologue.py")
PINS = os.path.join(ROOT, "tests", "test_prologue_oracle_pins.py")

MUTANTS = {
    # the kernel is applied forward in time (tap i on the token i steps back)
    "conv_taps_reversed": ("y[:, i:] += x[:, :T - i] * w[None, None, :, :, W - 1 - i]",
                           "y[:, i:] += x[:, :T - i] * w[None, None, :, :, i]"),
    # the convolution reads one token too far back
    "conv_shifted": ("y[:, i:] += x[:, :T - i] * w[None, None, :, :, W - 1 - i]",
                     "y[:, i + 1:] += x[:, :T - i - 1] * w[None, None, :, :, W - 1 - i]"),
    # eps added outside the square root
    "l2_eps_outside": ("return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)",
                       "return x / (np.sqrt(np.sum(x * x, axis=-1, keepdims=True)) + eps)"),
    # sigmoid of -x
    "sigmoid_sign": ("return 0.5 * (1.0 + np.tanh(0.5 * x))", "return 0.5 * (1.0 - np.tanh(0.5 * x))"),
    # SiLU without its factor x
    "silu_no_x": ("return x * sigmoid(x)", "return sigmoid(x)"),
    # softplus as a plain ReLU
    "softplus_relu": ("return np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x)))", "return np.maximum(x, 0.0)"),
    # the decay gate loses its minus sign (log alpha > 0)
    "gate_sign": ("return -a[None, None, :] * softplus(z + b[None, None, :])",
                  "return a[None, None, :] * softplus(z + b[None, None, :])"),
    # RMSNorm with the sum of squares instead of their mean
    "rms_sum": ("rs = 1.0 / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)",
                "rs = 1.0 / np.sqrt(np.sum(o * o, axis=-1, keepdims=True) + eps)"),
    # the output gate as a sigmoid instead of SiLU
    "gate_sigmoid": ("return o * rs * _f64(weight) * silu(g)", "return o * rs * _f64(weight) * sigmoid(g)"),
    # v without its activation
    "v_no_silu": ("v = silu(short_conv(v_in, conv_v))", "v = short_conv(v_in, conv_v)"),
    # v normalised like q and k
    "v_normalised": ("v = silu(short_conv(v_in, conv_v))", "v = l2_normalize(silu(short_conv(v_in, conv_v)), eps)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    pkg = tmp_path / "oracle"
    pkg.mkdir()
    (pkg / "__init__.py").write_text("")
    (pkg / "prologue.py").write_text(src.replace(old, new))
    shutil.copy(PINS, tmp_path / "test_pins.py")
    env = dict(os.environ, PYTHONPATH=str(tmp_path))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", "test_pins.py"],
                       cwd=tmp_path, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"


def test_unmutated_copy_passes(tmp_path):
    """The harness itself: the same copy without a mutation passes the pins."""
    pkg = tmp_path / "oracle"
    pkg.mkdir()
    (pkg / "__init__.py").write_text("")
    shutil.copy(SRC, pkg / "prologue.py")
    shutil.copy(PINS, tmp_path / "test_pins.py")
    env = dict(os.environ, PYTHONPATH=str(tmp_path))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", "test_pins.py"],
                       cwd=tmp_path, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-2000:]
