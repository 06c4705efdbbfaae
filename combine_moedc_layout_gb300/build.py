"""Build libmoedc.so in-tree with nvcc for sm_103a (no torch extension machinery).

Each translation unit compiles in parallel; the shared library lands in
combine_moedc_layout_gb300/_build/libmoedc.so.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(OUT_DIR, "libmoedc.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoedc")


def _sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps() -> list[str]:
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          out_dir: str | None = None) -> str:
    """Compile every csrc/*.cu and link libmoedc.so; returns its path.

    extra_flags / out_dir build a variant (for example with a tuning macro
    set by -D) into another directory without touching the default library."""
    if not force and not extra_flags and out_dir is None and up_to_date():
        return LIB_PATH
    OUT_DIR_ = out_dir or OUT_DIR
    LIB_PATH_ = os.path.join(OUT_DIR_, "libmoedc.so")
    os.makedirs(OUT_DIR_, exist_ok=True)
    nvcc = _nvcc()
    flags = ARCH + NVCC_FLAGS + (extra_flags or []) + ["-I" + INCLUDE, "-I" + CSRC]

    def compile_one(src: str) -> str:
        obj = os.path.join(OUT_DIR_, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = LIB_PATH_ + f".{os.getpid()}.tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH_)
    return LIB_PATH_


if __name__ == "__main__":
    print(build(force=True, verbose=True))
