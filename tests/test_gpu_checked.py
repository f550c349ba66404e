"""The bounds-checked build (-DMR_CHECKED): every gather index, row offset,
CSR row pointer and scatter destination that a kernel derives from data is
range-checked, a failed check skips its access and counts in a device error
word. The parity suites (seeded fuzz, every workload at full size, the
sort and maskedSelect forms, the ScheduleContext, permute and MoeUpdateExpert
operations) run against that build in a child process; each test must still
match the oracle bit for bit (or within the stated tolerance) and end with no
failed check (tests/conftest.py reads the words after every test). Only valid
inputs are used: no case makes an access fail on purpose."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SUITES = ["test_gpu_batching.py", "test_gpu_fuzz.py", "test_gpu_unpermute.py", "test_gpu_roundtrip.py",
          "test_gpu_context.py", "test_gpu_permute.py", "test_gpu_full_tail.py", "test_gpu_update_expert.py"]


def test_parity_suites_on_the_checked_build():
    from unpermute_stable_counting_gb300 import _build
    import __graft_entry__
    __graft_entry__.build()
    _build.build_library(checked=True)
    env = dict(os.environ, USC_CHECKED="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-m", "gpu", "-x", "-q", "-p", "no:cacheprovider"]
                       + [os.path.join("tests", f) for f in SUITES],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=3000)
    tail = r.stdout[-4000:] + r.stderr[-2000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and " failed" not in r.stdout, tail


def test_regular_build_has_no_checks():
    from unpermute_stable_counting_gb300 import _native
    if _native.checked_requested():
        pytest.skip("this process runs against the checked build")
    assert _native.checked_errors() is None
