"""Build libssd.so for sm_103a with nvcc (translation units compiled in parallel), and the
checked build libssd_checked.so (-DSSD_CHECKS=1: device-side index tests, for tests and
debugging).

    python -m speculative_decoding_copy_gb300.build [--verbose-ptxas] [--checked]

Objects go to speculative_decoding_copy_gb300/_build/ (_build_checked/), the libraries to
speculative_decoding_copy_gb300/lib/. Nothing here needs a GPU.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libssd.so")
LIB_CHECKED = os.path.join(LIBDIR, "libssd_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _compile(src: str, verbose_ptxas: bool, checked: bool = False) -> tuple[str, str]:
    obj = os.path.join(BUILD + ("_checked" if checked else ""), os.path.basename(src).replace(".cu", ".o"))
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "-I", os.path.join(ROOT, "include"), "-I", CSRC, "-c", src, "-o", obj]
    if checked:
        cmd.insert(1, "-DSSD_CHECKS=1")
    if verbose_ptxas:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(verbose_ptxas: bool = False, quiet: bool = True, checked: bool = False) -> str:
    bdir, lib = (BUILD + "_checked", LIB_CHECKED) if checked else (BUILD, LIB)
    os.makedirs(bdir, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose_ptxas, checked), srcs))
    objs = [o for o, _ in results]
    if verbose_ptxas and not quiet:
        for _, log in results:
            sys.stderr.write(log)
    tmp = lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build_all() -> tuple[str, str]:
    """Both libraries, built side by side."""
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        a = ex.submit(build)
        b = ex.submit(build, False, True, True)
        return a.result(), b.result()


if __name__ == "__main__":
    path = build(verbose_ptxas="--verbose-ptxas" in sys.argv, quiet=False, checked="--checked" in sys.argv)
    print(path)
