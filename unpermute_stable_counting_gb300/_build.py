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
# the bounds-checked build (-DMR_CHECKED): its own objects, library and stamp
CHECKED_FLAGS = ["-DMR_CHECKED"]
CHECKED_BUILD_DIR = os.path.join(CSRC, "_build_checked")
CHECKED_LIB_PATH = os.path.join(PKG, "libmoe_reorder_checked.so")
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


def _paths(checked: bool):
    if checked:
        return CHECKED_LIB_PATH, CHECKED_LIB_PATH + ".sha256", CHECKED_BUILD_DIR, CHECKED_FLAGS
    return LIB_PATH, STAMP_PATH, BUILD_DIR, []


def needs_build(extra_flags=None, checked: bool = False) -> bool:
    lib_path, stamp, _, cflags = _paths(checked)
    if not os.path.exists(lib_path) or not os.path.exists(stamp):
        return True
    with open(stamp) as f:
        return f.read().strip() != current_digest(cflags + list(extra_flags or []))


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


def build_library(force: bool = False, extra_flags: list[str] | None = None, checked: bool = False) -> str:
    """Build (or reuse) the library; checked=True builds the bounds-checked
    variant (-DMR_CHECKED) into its own objects and library file."""
    lib_path, _, _, cflags = _paths(checked)
    flags = cflags + list(extra_flags or [])
    if not force and not needs_build(extra_flags, checked):
        print(f"{os.path.basename(lib_path)}: reused (sources unchanged, digest "
              f"{current_digest(flags)[:16]})", file=sys.stderr)
        return lib_path
    with _build_lock():
        if not force and not needs_build(extra_flags, checked):
            return lib_path
        return _build_locked(extra_flags, checked)


def _build_locked(extra_flags: list[str] | None, checked: bool = False) -> str:
    lib_path, stamp, build_dir, cflags = _paths(checked)
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    flags = NVCC_FLAGS + cflags + list(extra_flags or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc] + flags + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj

    with fut.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH_FLAGS + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    digest = current_digest(cflags + list(extra_flags or []))
    os.replace(tmp, lib_path)
    with open(stamp + f".tmp{os.getpid()}", "w") as f:
        f.write(digest + "\n")
    os.replace(stamp + f".tmp{os.getpid()}", stamp)
    print(f"{os.path.basename(lib_path)}: compiled (digest {digest[:16]})", file=sys.stderr)
    return lib_path


if __name__ == "__main__":
    print(build_library(force=True))
