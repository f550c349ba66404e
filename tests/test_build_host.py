"""Host-only checks of the build's reuse decision: the CUDA library and the
oracle are rebuilt when their sources' contents (or the flags) differ from
the stamp written at the last build, never on file times alone."""
import os
import time

import pytest

from unpermute_stable_counting_gb300 import _build


def test_digest_follows_content_and_flags_not_times(tmp_path):
    a = tmp_path / "a.cu"
    b = tmp_path / "b.cuh"
    a.write_text("int x;\n")
    b.write_text("int y;\n")
    files = [str(a), str(b)]
    d0 = _build.source_digest(files, ["-O3"], "nvcc 13.0", "x86_64")
    os.utime(a, (time.time() + 100, time.time() + 100))   # newer time, same content
    assert _build.source_digest(files, ["-O3"], "nvcc 13.0", "x86_64") == d0
    a.write_text("int x = 1;\n")                           # new content
    d1 = _build.source_digest(files, ["-O3"], "nvcc 13.0", "x86_64")
    assert d1 != d0
    assert _build.source_digest(files, ["-O2"], "nvcc 13.0", "x86_64") != d1   # flags
    assert _build.source_digest(files, ["-O3"], "nvcc 13.0", "aarch64") != d1  # machine
    assert _build.source_digest(files, ["-O3"], "nvcc 13.1", "x86_64") != d1   # compiler


def test_library_stamp_decides_reuse():
    _build.build_library()
    assert not _build.needs_build()
    with open(_build.STAMP_PATH) as f:
        good = f.read()
    try:
        with open(_build.STAMP_PATH, "w") as f:
            f.write("0" * 64 + "\n")                       # a binary from other sources
        assert _build.needs_build()
    finally:
        with open(_build.STAMP_PATH, "w") as f:
            f.write(good)
    assert not _build.needs_build()
    assert _build.needs_build(["-DSOME_OTHER_FLAG"])      # other flags: other digest


def test_oracle_stamp_decides_reuse():
    oracle = pytest.importorskip("oracle")
    oracle.build()
    assert not oracle._stale()
    stamp = oracle._LIB + ".sha256"
    with open(stamp) as f:
        good = f.read()
    try:
        with open(stamp, "w") as f:
            f.write("0" * 64 + "\n")
        assert oracle._stale()
    finally:
        with open(stamp, "w") as f:
            f.write(good)
    assert not oracle._stale()
