"""Build libmxq.so (and its --use_fast_math twin) in-tree with nvcc for sm_103a.

    python -m block_scaled_precision_x32_gb300.build [--force]

Each translation unit compiles in parallel, then one nvcc link makes the
shared library under ``block_scaled_precision_x32_gb300/_build/``.  The fast-math
twin exists only so the tests can show that the bytes do not depend on it.
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
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
BASE_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "-I", INCLUDE, "-I", CSRC]

VARIANTS = {
    "libmxq.so": [],
    "libmxq_fastmath.so": ["--use_fast_math"],
}


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmxq")
    return cand


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs_mtime() -> float:
    files = sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
    files += [os.path.join(INCLUDE, "mxq.h"), os.path.abspath(__file__)]
    return max(os.path.getmtime(f) for f in files)


def lib_path(name: str = "libmxq.so") -> str:
    return os.path.join(BUILD, name)


def _compile(src: str, obj: str, extra):
    cmd = [nvcc()] + ARCH + BASE_FLAGS + list(extra) + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stderr


def build(force: bool = False, verbose: bool = False) -> dict:
    """Compile every variant that is missing or older than its sources."""
    os.makedirs(BUILD, exist_ok=True)
    newest = _inputs_mtime()
    todo = [name for name in VARIANTS
            if force or not os.path.exists(lib_path(name)) or os.path.getmtime(lib_path(name)) < newest]
    if todo:
        jobs = []
        with cf.ThreadPoolExecutor(max_workers=min(16, (os.cpu_count() or 4))) as ex:
            for name in todo:
                tag = name.replace(".so", "")
                for src in sources():
                    obj = os.path.join(BUILD, f"{tag}.{os.path.basename(src)}.o")
                    jobs.append((name, obj, ex.submit(_compile, src, obj, VARIANTS[name])))
            for _, _, fut in jobs:
                msg = fut.result()
                if verbose and msg:
                    print(msg, file=sys.stderr)
        for name in todo:
            objs = [obj for n, obj, _ in jobs if n == name]
            tmp = lib_path(name) + f".tmp{os.getpid()}"
            cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-cudart", "static"]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
            os.replace(tmp, lib_path(name))
    return {name: lib_path(name) for name in VARIANTS}


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
