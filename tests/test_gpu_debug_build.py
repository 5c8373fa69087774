"""The sanitizer substitute (guard regions around every output, and the debug library's
device-side index checks), run through each library variant in a process of its own: the
release library (libmsa.so) and the debug library (libmsa_debug.so, built with -DMSA_DEBUG
on first use).  The two export the same symbols and device variables, so one process loads
one of them.
The cases are in tests/debug_build_cases.py."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
@pytest.mark.parametrize("variant", ["release", "debug"])
def test_guarded_cases(variant):
    env = dict(os.environ, MSA_LIBRARY_VARIANT=variant)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join("tests", "debug_build_cases.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
