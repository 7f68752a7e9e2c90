"""Build libawq.so in-tree with nvcc for sm_103a.

    python -m post_weight_quantization_33_b300.build [--force] [--verbose] [--checked]

Every .cu file under csrc/ is compiled separately (in parallel) with
``-gencode arch=compute_103a,code=sm_103a`` and linked into one shared
library next to this file.  ``--checked`` builds libawq_checked.so instead:
the same sources with -DAWQ_CHECK_BOUNDS, whose kernels check their computed
global indexes against the buffers' extents (awq_bounds_report).  The CUDA runtime is linked statically, and the
driver's tensor-map encoder is looked up at run time, so the library loads
(and exports its symbols) on a machine without a GPU driver.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libawq.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)
CHECKED_BUILD_DIR = os.path.join(PKG, "_build_checked")
CHECKED_LIB_PATH = os.path.join(PKG, "libawq_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-Xptxas", "-v", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libawq")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    hs.append(os.path.join(INCLUDE, "awq.h"))
    return hs


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, verbose: bool, checked: bool = False) -> tuple[str, str]:
    obj = os.path.join(CHECKED_BUILD_DIR if checked else BUILD_DIR, os.path.basename(src) + ".o")
    cmd = [nvcc(), "-c", src, "-o", obj] + ARCH + NVCC_FLAGS
    if checked:
        cmd += ["-DAWQ_CHECK_BOUNDS"]
    if os.path.basename(src) == "awq_api.cu":
        cmd += ["-Xcompiler", "-fvisibility=default"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
    if verbose:
        sys.stderr.write(res.stderr)
    return obj, res.stderr


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compile and link libawq.so (or, with ``checked``, libawq_checked.so)
    if any source is newer; return its path."""
    lib_path = CHECKED_LIB_PATH if checked else LIB_PATH
    srcs = sources()
    deps = srcs + headers()
    if not force and not _stale(lib_path, deps):
        return lib_path
    os.makedirs(CHECKED_BUILD_DIR if checked else BUILD_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = [f.result()[0] for f in [ex.submit(_compile, s, verbose, checked) for s in srcs]]
    tmp = lib_path + ".tmp"
    cmd = [nvcc(), "-shared", "-o", tmp] + objs + ARCH + ["-Xcompiler", "-fPIC"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--checked", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, checked=a.checked))
