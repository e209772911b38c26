"""Build libssdscan.so in-tree with nvcc for sm_103a (no cmake, no torch extension machinery).

Each .cu under csrc/ is compiled in parallel to an object under _build/, then linked into
chunked_ssd_scan_gb300/libssdscan.so.  The build is skipped when the library is newer than every
source and header.  `build_checked()` makes the index-checked debug library
(libssdscan_checked.so: every checked output access that would fall outside its buffer is
skipped and latches SSD_ERR_INDEX in the workspace) from the same sources.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libssdscan.so")
LIB_CHECKED = os.path.join(PKG, "libssdscan_checked.so")
BUILD_CHECKED = os.path.join(PKG, "_build_checked")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"]


def _nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(ROOT, "include", "*.h")) + [os.path.abspath(__file__)])


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=(), lib: str = LIB,
          build_dir: str = BUILD) -> str:
    if not force and up_to_date(lib):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    srcs = _sources()

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra_flags, "-I", os.path.join(ROOT, "include"), "-c",
               src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build_checked(force: bool = False) -> str:
    """The index-checked debug library (same sources, compiled with SSD_INDEX_CHECKS)."""
    return build(force=force, extra_flags=("-DSSD_INDEX_CHECKS",), lib=LIB_CHECKED,
                 build_dir=BUILD_CHECKED)


if __name__ == "__main__":
    print(build(force=True, verbose=True))
