"""The pins are strong enough: each plausible mistake, planted in a copy of the
oracle on the CPU, makes tests/test_oracle_pins.py fail.  The unmodified copy
passes.  No GPU is involved."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

# (what the mistake is, text in oracle/__init__.py, replacement)
MUTATIONS = [
    ("smoothing mass over V-1 classes", "dz = g[:, None] * (p - eps / vocab)",
     "dz = g[:, None] * (p - eps / (vocab - 1))"),
    ("smoothing term dropped from the loss",
     "loss[rows] += eps * (lse[rows] - z[rows].sum(axis=1) / vocab)", "pass"),
    ("wrong sign of the target term", "dz -= np.where(hit", "dz += np.where(hit"),
    ("dW off by a scale", "return dz @ wd, dz.T @ xd, dz", "return dz @ wd, (xd.T @ dz).T * 1.0001, dz"),
    ("mean over all rows instead of non-ignored",
     "return np.full(n, grad_output[0] / n_valid)", "return np.full(n, grad_output[0] / n)"),
    ("log-sum-exp perturbed", "lse = m + np.log(np.exp(z - m[:, None]).sum(axis=1))",
     "lse = m + np.log(np.exp(z - m[:, None]).sum(axis=1) + 1e-9)"),
    ("target index off by one", "zy = z[rows, np.asarray(target)[rows]]",
     "zy = z[rows, np.asarray(target)[rows] - 1]"),
    ("ignored rows keep their statistics", "m = np.where(ignored, 0.0, m)", "m = m"),
    ("sum reduction divides by N_v", "        return np.full(n, grad_output[0])\n",
     "        return np.full(n, grad_output[0] / max(n_valid, 1))\n"),
    ("entropy sign flipped", "return lse - (p * z).sum(axis=1)", "return lse + (p * z).sum(axis=1)"),
]


def _run_pins_against(tmp_path, source: str) -> int:
    pkg = tmp_path / "oracle"
    if pkg.exists():
        shutil.rmtree(pkg)
    pkg.mkdir()
    (pkg / "__init__.py").write_text(source)
    env = dict(os.environ, PYTHONPATH=f"{tmp_path}{os.pathsep}{ROOT}")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", PINS],
                       cwd=str(tmp_path), env=env, capture_output=True, text=True, timeout=600)
    return r.returncode


@pytest.fixture(scope="module")
def source():
    with open(os.path.join(ROOT, "oracle", "__init__.py")) as f:
        return f.read()


def test_unmodified_copy_passes(tmp_path, source):
    assert _run_pins_against(tmp_path, source) == 0


@pytest.mark.parametrize("what,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, source, what, old, new):
    assert old in source, f"mutation site missing: {what}"
    assert _run_pins_against(tmp_path, source.replace(old, new, 1)) != 0, what
