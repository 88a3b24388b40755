"""The bounds-checked debug build (-DMLA_CHECKS).

Compute-sanitizer is not available for these kernels' runs, so the library
carries its own checks: built with -DMLA_CHECKS, every kernel tests its ring
slots, TMEM columns, swizzled shared-memory offsets, histogram bins and
output positions, and a failed check records MLA_ERR_CHECK (with the file
and line) in the device status instead of trapping.  This test builds that
variant and runs the small parity cases against it in a child process
(tests/checks_cases.py): no check may fail and every output must still match
the fp64 oracle.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def test_checked_build_reports_no_violation_on_the_parity_cases():
    from mla_family_attention_gb300.build import build
    lib = build(checks=True)
    env = dict(os.environ, MLA_GB300_LIB=lib)
    r = subprocess.run([sys.executable, os.path.join(HERE, "checks_cases.py")], env=env,
                       capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, (r.stdout[-3000:], r.stderr[-3000:])
    assert "checked cases ok" in r.stdout
