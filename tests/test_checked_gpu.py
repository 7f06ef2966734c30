"""The checked build of libciera (-DCIERA_CHECKED): every global access at a
computed offset is tested against its buffer, and one that would leave it is
skipped and reported as CIERA_E_BOUNDS instead of touching memory.

The GPU parity suites (small, random and full-size cases, graphs, the
pipeline, the allocation-free entry point) run once more in a child process against the
checked library (CIERA_CHECKED=1), which must give the same bytes and no
status; the test hook CIERA_DEBUG_OUT_OF_RANGE, accepted only by the checked
build, shows that the checks fire and that the library recovers."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from lossless_exponent_reuse_gb300 import ciera
from lossless_exponent_reuse_gb300.allgather import SimulatedAllgather

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
         "tests/test_random_gpu.py",
         "tests/test_checked_gpu.py::test_out_of_range_hook_is_caught",
         "tests/test_zz_no_alloc.py"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and " skipped" not in r.stdout.splitlines()[-1], r.stdout[-500:]


def _bf16(rng, n):
    x = rng.normal(0.0, 0.02, n).astype(np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def test_out_of_range_hook_is_caught():
    if not ciera.checked_build():
        pytest.skip("the hook exists in the checked build only")
    assert ciera.library_path().endswith("libciera_checked.so")
    n, R, B = 131072, 4, 256
    rng = np.random.default_rng(4)
    w0 = _bf16(rng, n)
    w1 = w0.copy()
    w1[::5000] ^= np.uint16(0x0080)                  # a few changed blocks: COMPRESSED
    dev = lambda w: torch.from_numpy(w.view(np.int16)).cuda().view(torch.uint16)
    ag = SimulatedAllgather(n, B, R)
    ag.step(dev(w0))
    assert ag.status() == ciera.OK
    ag.plan.compress(dev(w1), ag.sender_cache, ag.payloads, ag.descs, ag.workspace,
                     extra_flags=ciera.DEBUG_OUT_OF_RANGE)
    assert ag.status() == ciera.E_BOUNDS
    # a cold start re-seeds both sides; the library is usable again
    ag.iteration = 0
    out = ag.step(dev(w1))
    assert ag.status() == ciera.OK
    np.testing.assert_array_equal(out[:n].view(torch.int16).cpu().numpy().view(np.uint16), w1)
