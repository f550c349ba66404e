import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: larger CPU cases")


@pytest.fixture(autouse=True)
def _checked_build_words(request):
    """In a run against the bounds-checked library (USC_CHECKED=1), every GPU
    test must end with no failed bounds check."""
    yield
    if os.environ.get("USC_CHECKED") != "1" or request.node.get_closest_marker("gpu") is None:
        return
    import torch
    if not torch.cuda.is_available():
        return
    from unpermute_stable_counting_gb300 import _native
    res = _native.checked_errors(reset=True)
    assert res is not None, "USC_CHECKED=1 but the loaded library is not the checked build"
    assert res[0] == 0, f"{res[0]} bounds checks failed (the first at site {res[1]})"
