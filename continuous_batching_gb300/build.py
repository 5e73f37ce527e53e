"""Builds libpagedattn.so in-tree with nvcc for sm_103a (no CMake, no torch extension).

    python -m continuous_batching_gb300.build          # incremental
    python -m continuous_batching_gb300.build --force  # rebuild everything

Each translation unit compiles in parallel to continuous_batching_gb300/_build/*.o, then one
link step produces continuous_batching_gb300/libpagedattn.so (CUDA runtime linked statically,
so the library needs only the NVIDIA driver at run time).
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libpagedattn.so")
HEADERS = [os.path.join(ROOT, "include", "pagedattn.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O3",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]
SOURCES = ["host.cpp", "sched.cpp", "pipeline.cpp", "kv_write.cu", "attention.cu"]


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpagedattn")
    return p


def _deps() -> list:
    out = list(HEADERS)
    for f in os.listdir(CSRC):
        if f.endswith(".h"):
            out.append(os.path.join(CSRC, f))
    return out


def _stale(target: str, sources: list) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in sources)


# what the last build() in this process did: the translation units it compiled (the others were
# up to date) and whether it linked the library
LAST_BUILD = {}


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    deps = _deps()
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src + ".o")
        objs.append(o)
        if force or _stale(o, [s] + deps):
            extra = ["-x", "cu"] if src.endswith(".cu") else []
            jobs.append([cc] + ARCH + FLAGS + extra + ["-c", s, "-o", o])

    def run(cmd):
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, flush=True)

    with ThreadPoolExecutor(max_workers=max(1, len(jobs))) as ex:
        list(ex.map(run, jobs))
    linked = bool(force or jobs or _stale(LIB, objs))
    if linked:
        tmp = LIB + ".tmp"
        run([cc] + ARCH + ["-shared", "-o", tmp] + objs)
        os.replace(tmp, LIB)
    LAST_BUILD.clear()
    LAST_BUILD.update(compiled=[os.path.basename(j[-3]) for j in jobs], linked=linked,
                      arch=" ".join(ARCH), library=LIB)
    return LIB


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-v", "--verbose", action="store_true")
    a = ap.parse_args(argv)
    print(build(force=a.force, verbose=a.verbose))
    return 0


if __name__ == "__main__":
    sys.exit(main())
