"""The GPU suite again, against the checked build (libfa_checked.so, built
with FA_DEBUG_CHECKS).  Its kernels check every plain global load and store
against the extent the call's arguments give its buffer.  A failing access
is skipped and sets FA_DEV_BAD_INDEX rather than faulting, and the autouse
fixture in conftest.py fails any test that leaves that bit set.  The checks
stand in for a memory checker on this pool.  TMA copies are bounded by their
tensor maps and need none."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(os.environ.get("FA_CHECKED") == "1", reason="already the checked run")
def test_gpu_suite_under_checked_build():
    from exact_attention_33_gb300.build import build
    build()
    build(checked=True)
    env = dict(os.environ, FA_CHECKED="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "tests", "-m", "gpu", "-x", "-q",
                        "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                       text=True, timeout=1800)
    tail = "\n".join(r.stdout.strip().splitlines()[-25:])
    assert r.returncode == 0, "GPU suite failed under the checked build:\n" + tail
    assert " passed" in tail
