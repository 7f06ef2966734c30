"""The checked build of libciera (-DCIERA_CHECKED): every global access at a
computed offset is tested against its buffer, and one that would leave it is
skipped and reported as CIERA_E_BOUNDS instead of touching memory.

The GPU parity suites (small, random and full-size cases, graphs, the
pipeline, the receiver over separate payload buffers and the host-buffer
step, the allocation-free entry point) run once more in a child process against the
checked library (CIERA_CHECKED=1), which must give the same bytes and no
status."""
import os
import subprocess
import sys

import pytest

from lossless_exponent_reuse_gb300 import ciera

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def test_parity_suites_under_the_checked_build():
    if ciera.checked_build():
        pytest.skip("already inside the checked build")
    env = dict(os.environ, CIERA_CHECKED="1")
    r = subprocess.run(
        [sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider",
         "tests/test_parity_gpu.py", "tests/test_hashed_gpu.py", "tests/test_rans_gpu.py",
         "tests/test_fullsize_gpu.py", "tests/test_graph_gpu.py", "tests/test_pipeline_gpu.py",
         "tests/test_random_gpu.py", "tests/test_gather_host_gpu.py",
         "tests/test_zz_no_alloc.py"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and " skipped" not in r.stdout.splitlines()[-1], r.stdout[-500:]
