"""The bounds-checked debug build (-DSPEC_CHECKED) on the GPU.

The parity suites of every kernel run again in a child process with
SPEC_TREE_CHECKED=1, so that every entry point loads libspec_tree_checked.so
(the suites' session fixture asserts which build it loaded).  On valid inputs
no index check may fire: the suites' status words stay 0 and every result
matches the oracle as in the normal build.  The malformed-input cases of the
suites still get their own codes (a check skips only accesses outside the
call's buffers, which those inputs never reach)."""
import glob
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# every GPU suite but this one; collected after them, so that a run stopping
# at the first failure has run the normal build's suites first
SUITES = sorted(os.path.relpath(p, ROOT) for p in glob.glob(os.path.join(ROOT, "tests", "test_gpu_*.py")))
SUITES.append("tests/test_zz_no_alloc.py")


@pytest.mark.gpu
def test_parity_suites_pass_on_the_bounds_checked_build(gpu_lib):
    from token_tree_verification_gb300 import build
    build.build(checked=True)
    env = dict(os.environ, SPEC_TREE_CHECKED="1")
    # the million-trial chi-square runs measure statistics the normal build
    # already covers; the rest of each suite runs
    cmd = [sys.executable, "-m", "pytest", *SUITES, "-m", "gpu", "-x", "-q", "-p", "no:cacheprovider",
           "-k", "not chi_square"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    tail = "\n".join((r.stdout + r.stderr).splitlines()[-25:])
    assert r.returncode == 0, tail
    assert " passed" in tail and "failed" not in tail, tail
