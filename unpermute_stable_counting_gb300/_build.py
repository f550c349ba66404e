"""Build the CUDA library libmoe_reorder.so in-tree for sm_103a (GB300).

Each translation unit under csrc/ is compiled in parallel with nvcc, then
linked into one shared library next to this file. No torch headers are
involved: the library's ABI is plain C (include/moe_reorder.h).

Whether a build is needed is decided by content, not file times: the library
is stamped with a SHA-256 digest of every source and header it is built from,
the nvcc flags, the compiler's version and the host machine type, and it is
rebuilt whenever the stamp is missing or differs. A binary copied in with a
newer time but from other sources is therefore never reused.
"""
from __future__ import annotations

import concurrent.futures as fut
import contextlib
import fcntl
import glob
import hashlib
import os
import platform
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD_DIR = os.path.join(CSRC, "_build")
LIB_PATH = os.path.join(PKG, "libmoe_reorder.so")
STAMP_PATH = LIB_PATH + ".sha256"
HEADER = os.path.join(ROOT, "include", "moe_reorder.h")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH_FLAGS + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                           "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [HEADER, __file__]


def _nvcc_version() -> str:
    try:
        r = subprocess.run([_nvcc(), "--version"], capture_output=True, text=True)
        return r.stdout.strip().splitlines()[-1] if r.stdout.strip() else ""
    except OSError:
        return ""


def source_digest(files, flags, tool_version: str = "", machine: str = "") -> str:
    """SHA-256 over the files' names (relative to the repository) and contents,
    the flags, the compiler version and the machine type."""
    h = hashlib.sha256()
    for f in sorted(files):
        h.update(os.path.relpath(f, ROOT).encode() + b"\0")
        with open(f, "rb") as fh:
            h.update(fh.read())
        h.update(b"\0")
    for x in list(flags) + [tool_version, machine]:
        h.update(str(x).encode() + b"\0")
    return h.hexdigest()


def current_digest(extra_flags=None) -> str:
    return source_digest(_deps(), NVCC_FLAGS + list(extra_flags or []), _nvcc_version(),
                         platform.machine())


def needs_build(extra_flags=None) -> bool:
    if not os.path.exists(LIB_PATH) or not os.path.exists(STAMP_PATH):
        return True
    with open(STAMP_PATH) as f:
        return f.read().strip() != current_digest(extra_flags)


@contextlib.contextmanager
def _build_lock():
    """One builder at a time (parallel test workers share the tree)."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    with open(os.path.join(BUILD_DIR, ".lock"), "w") as f:
        fcntl.flock(f, fcntl.LOCK_EX)
        try:
            yield
        finally:
            fcntl.flock(f, fcntl.LOCK_UN)


def build_library(force: bool = False, extra_flags: list[str] | None = None) -> str:
    if not force and not needs_build(extra_flags):
        print(f"libmoe_reorder.so: reused (sources unchanged, digest {current_digest(extra_flags)[:16]})",
              file=sys.stderr)
        return LIB_PATH
    with _build_lock():
        if not force and not needs_build(extra_flags):
            return LIB_PATH
        return _build_locked(extra_flags)


def _build_locked(extra_flags: list[str] | None) -> str:
    nvcc = _nvcc()
    flags = NVCC_FLAGS + list(extra_flags or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD_DIR, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc] + flags + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj

    with fut.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH_FLAGS + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    digest = current_digest(extra_flags)
    os.replace(tmp, LIB_PATH)
    with open(STAMP_PATH + f".tmp{os.getpid()}", "w") as f:
        f.write(digest + "\n")
    os.replace(STAMP_PATH + f".tmp{os.getpid()}", STAMP_PATH)
    print(f"libmoe_reorder.so: compiled (digest {digest[:16]})", file=sys.stderr)
    return LIB_PATH


if __name__ == "__main__":
    print(build_library(force=True))
