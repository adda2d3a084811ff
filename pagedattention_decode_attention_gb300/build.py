"""Builds ``libpagedattn.so`` in-tree with nvcc for sm_103a.

Each translation unit compiles in parallel, then one link step makes the shared
library next to this file.  The CUDA runtime is linked statically, so the
library loads on a machine without a GPU (the pool and symbol tests need that)
and on a GPU machine alongside PyTorch's own runtime.

    python -m pagedattention_decode_attention_gb300.build [--force] [--verbose]
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
LIB_NAME = "libpagedattn.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["status.cpp", "pool.cpp", "tensor_map.cpp", "copy_kernels.cu", "decode.cu", "prefill.cu"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpagedattn.so")


def _flags(src: str) -> list[str]:
    common = ["-O3", "-std=c++17", "-I", INCLUDE, "-I", CSRC,
              "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden"]
    if src.endswith(".cu"):
        # PA_NVCC_EXTRA adds flags for a diagnostic build, e.g. -DPA_PROFILE_TIMES
        # for the per-role wait counters (rebuild with --force to apply)
        extra = os.environ.get("PA_NVCC_EXTRA", "").split()
        return common + ARCH + ["-lineinfo", "--expt-relaxed-constexpr", "-Xptxas", "-v"] + extra
    return common + ["-x", "c++"]


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _headers() -> list[str]:
    hs = [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    hs += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return hs


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if stale) and return the path of the shared library."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    tool = nvcc()
    headers = _headers()
    jobs = []
    for src in SOURCES:
        src_path = os.path.join(CSRC, src)
        obj = os.path.join(BUILD_DIR, src + ".o")
        if force or _stale(obj, [src_path] + headers):
            jobs.append((src, [tool, "-c", src_path, "-o", obj] + _flags(src)))

    def run(job):
        name, cmd = job
        res = subprocess.run(cmd, capture_output=True, text=True)
        return name, cmd, res

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        for name, cmd, res in ex.map(run, jobs):
            if verbose or res.returncode != 0:
                sys.stderr.write(f"[build] {' '.join(cmd)}\n{res.stdout}{res.stderr}")
            if res.returncode != 0:
                raise RuntimeError(f"nvcc failed on {name}")

    objs = [os.path.join(BUILD_DIR, s + ".o") for s in SOURCES]
    if force or jobs or _stale(LIB_PATH, objs):
        tmp = LIB_PATH + ".tmp"
        cmd = [tool, "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "static"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or res.returncode != 0:
            sys.stderr.write(f"[build] {' '.join(cmd)}\n{res.stdout}{res.stderr}")
        if res.returncode != 0:
            raise RuntimeError("link of libpagedattn.so failed")
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose))


if __name__ == "__main__":
    main()
