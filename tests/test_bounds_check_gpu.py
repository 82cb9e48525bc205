"""The bounds-checking build (-DVCE_BOUNDS_CHECK): every kernel checks the
addresses it computes and reports VCE_DEVSTATUS_BOUNDS instead of making an
access that fails.  It stands in for a memory checker, which cannot run on
this pool.  This test builds that variant, runs tests/bounds_cases.py against
it in a child process (the library is chosen when the package first loads it),
and requires every case to match the oracle with the status word zero."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bounds_build_exports_its_flag():
    # CPU: the checking variant compiles (nvcc cross-compiles without a GPU)
    from vocabulary_cross_entropy_gb300 import build
    lib = build.build_bounds_check()
    assert os.path.exists(lib) and lib != build.LIB


@pytest.mark.gpu
def test_every_kernel_passes_its_bounds_checks():
    from vocabulary_cross_entropy_gb300 import build
    lib = build.build_bounds_check()
    env = dict(os.environ, VCE_LIBRARY=lib)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "bounds_cases.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "bounds cases ok" in r.stdout
