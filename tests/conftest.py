import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: large CPU-side work")


@pytest.fixture(autouse=True)
def _checked_build_index_word(request):
    """Under FA_CHECKED=1 the binding loads the checked build, whose kernels
    check every plain global access against its buffer's extent and set
    FA_DEV_BAD_INDEX instead of making a bad one.  Every GPU test then also
    has to leave that bit clear."""
    yield
    if os.environ.get("FA_CHECKED") == "1" and request.node.get_closest_marker("gpu"):
        import exact_attention_33_gb300 as fa
        assert fa.library_path().endswith("libfa_checked.so")
        st = fa.fa_device_status(clear=False)
        assert st & fa.FA_DEV_BAD_INDEX == 0, f"{request.node.name}: a kernel index left its buffer"
